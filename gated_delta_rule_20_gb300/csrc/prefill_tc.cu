// prefill_tc.cu -- chunk-parallel prefill of the gated delta-rule recurrence on
// the 5th-generation tensor cores (tcgen05 + TMEM + TMA), bf16 operands with
// fp32 accumulation and an fp32 state.  Dk = Dv = 128, chunk C = 64.
//
// What it computes: the "GDN CTE Kernel API Reference" prefill (Parameters:
// q, k [B,Hk,S,Dk] token-major, v [B,Hv,S,Dv], g_log / beta [B,Hv,S] fp32,
// scale applied on device, optional in/out fp32 state; Returns: head-major
// un-normalised output in the compute dtype and the final fp32 state; Notes:
// value head h reads key head h / (Hv/Hk), the state stays fp32).
//
// Chunk algebra, for a chunk of C tokens with start state S0, G_r = cumulative
// log-decay inside the chunk, gamma_r = exp(G_r):
//     A[r][j] = beta_r exp(G_r - G_j) k_r.k_j  (j < r)        T = (I + A)^-1
//     U = T diag(beta) V,  W = T diag(beta gamma) K,  Delta = U - W S0
//     O = scale (diag(gamma) Q S0 + P Delta),  P[r][j] = exp(G_r - G_j) q_r.k_j (j <= r)
//     S_end = gamma_C S0 + sum_j exp(G_C - G_j) k_j Delta_j^T
// Only exponents <= 0 are ever evaluated, so strong decay cannot overflow.
//
// Orientation.  Every tensor-core product is issued with M = 128 by putting a
// head dimension (Dv or Dk = 128) on the M / TMEM-lane axis and the chunk's 64
// tokens on N:
//     R_KQ  = [K; Q] K^T          (lanes 0..63: K K^T rows, 64..127: Q K^T rows)
//     R_QS  = S0^T Q^T            (lanes = dv, columns = token r)
//     R_U   = V^T (T diag beta)^T               -> U^T
//     R_W   = K^T (T diag beta gamma)^T         -> W^T
//     R_U  += S0^T (-W)^T                       -> Delta^T
//     R_PD  = Delta^T P^T                       (reuses R_KQ's columns)
//     R_SN  = (Delta diag(exp(G_C - G)))^T K    -> increment of S^T
// The fp32 state lives in TMEM as S^T (lane = dv, column = dk); a bf16 copy in
// shared memory is the A operand of the two products that read S0.
// Thread i of the 128-thread CTA owns TMEM lane i (dv row i, or dk row i, or
// token row i of the Gram products), so every epilogue step is row-local.
//
// Structure: one CTA per (batch, value head); one thread issues TMA loads and
// MMAs; the chunk inputs (q, k, v tiles) are double-buffered so the next
// chunk's loads overlap this chunk's work.  Every wait is bounded; a wait that
// gives up records GDN_ERR_TIMEOUT in the device status word, drains what is in
// flight (again bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "gdn_internal.h"
#include "sm100_ptx.cuh"

namespace gdn {
namespace {

using namespace ptx;

constexpr int kC = 64;        // tokens per chunk
constexpr int kD = 128;       // Dk = Dv
constexpr int kThreads = 128;
constexpr uint32_t kTmemCols = 512;

// TMEM columns (fp32, 128 lanes each)
constexpr uint32_t COL_KQ = 0;    // 64: [K;Q] K^T, later Delta^T P^T
constexpr uint32_t COL_U = 64;    // 64: U^T, then Delta^T
constexpr uint32_t COL_W = 128;   // 64: W^T
constexpr uint32_t COL_QS = 192;  // 64: S0^T Q^T
constexpr uint32_t COL_SN = 256;  // 128: state increment (S^T layout)
constexpr uint32_t COL_S = 384;   // 128: fp32 state S^T

// Shared memory (bytes from a 1024-aligned base).  All bf16 tiles use rows of
// 128 bytes with the 128-byte swizzle.
constexpr uint32_t STAGE_BYTES = 49152;
constexpr uint32_t ST_K0 = 0;       // K, dk 0..63   [64 tokens][64]
constexpr uint32_t ST_Q0 = 8192;    // Q, dk 0..63
constexpr uint32_t ST_K1 = 16384;   // K, dk 64..127
constexpr uint32_t ST_Q1 = 24576;   // Q, dk 64..127
constexpr uint32_t ST_V0 = 32768;   // V, dv 0..63
constexpr uint32_t ST_V1 = 40960;   // V, dv 64..127
constexpr uint32_t OFF_T1 = 2 * STAGE_BYTES;  // T diag(beta)        [64 r][64 j] K-major
constexpr uint32_t OFF_T2 = OFF_T1 + 8192;    // T diag(beta gamma)  [64 r][64 j]
constexpr uint32_t OFF_P = OFF_T2 + 8192;     // P                   [64 r][64 j]
constexpr uint32_t OFF_WD = OFF_P + 8192;     // -W as [dk][64 r] (MN-major B), then Delta^T [dv][64 j]
constexpr uint32_t OFF_DT = OFF_WD + 16384;   // Delta~^T [dv][64 j]; fp32 T during the solve
constexpr uint32_t OFF_SB = OFF_DT + 16384;   // S^T bf16 [dv][dk]: dk halves at +0, +16384
constexpr uint32_t OFF_OUT = OFF_SB + 32768;  // out tile: dv halves at +0, +8192; fp32 A during the solve
constexpr uint32_t OFF_SMALL = OFF_OUT + 16384;  // G, gamma, beta, exp(G_C - G): 4 x 64 floats
constexpr uint32_t OFF_BAR = OFF_SMALL + 1024;   // 3 mbarriers, TMEM base, flags
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // slack for the 1024-byte alignment

static_assert(SMEM_ALLOC <= 232448, "shared memory budget");

// Instruction descriptors (M = 128 always).
constexpr uint32_t IDESC_N64_KK = make_idesc_bf16(128, 64, 0, 0);
constexpr uint32_t IDESC_N64_MK = make_idesc_bf16(128, 64, 1, 0);   // A MN-major
constexpr uint32_t IDESC_N64_KM = make_idesc_bf16(128, 64, 0, 1);   // B MN-major
constexpr uint32_t IDESC_N128_KM = make_idesc_bf16(128, 128, 0, 1);

// fp32 64x64 scratch with an XOR swizzle on the column: conflict-free row and
// column access.
__device__ __forceinline__ int fidx(int r, int c) { return r * 64 + (c ^ (r & 31)); }

// Write 32 fp32 values as bf16 into a 128-byte-swizzled row: bytes
// [byte0, byte0 + 64) of row `row` of the tile at `tile`.
__device__ __forceinline__ void st_row_bf16x32(uint8_t* tile, int row, int byte0, const float (&x)[32],
                                               float mul = 1.0f) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(x[8 * q + 0] * mul, x[8 * q + 1] * mul);
        w.y = pack_bf16x2(x[8 * q + 2] * mul, x[8 * q + 3] * mul);
        w.z = pack_bf16x2(x[8 * q + 4] * mul, x[8 * q + 5] * mul);
        w.w = pack_bf16x2(x[8 * q + 6] * mul, x[8 * q + 7] * mul);
        *reinterpret_cast<uint4*>(tile + sw128_offset(row, byte0 + 16 * q)) = w;
    }
}

struct Shared {
    uint8_t* base;
    uint32_t sbase;
    float* G;
    float* gam;
    float* bet;
    float* ec;
    uint64_t* bar_tma;  // [2]
    uint64_t* bar_mma;
    uint32_t* tmem_slot;
};

__device__ __forceinline__ void issue_chunk_loads(const Shared& sh, int stage, const CUtensorMap* tq,
                                                  const CUtensorMap* tk, const CUtensorMap* tv, int t0, int bhk,
                                                  int bh) {
    uint8_t* st = sh.base + stage * STAGE_BYTES;
    uint64_t* bar = &sh.bar_tma[stage];
    mbar_arrive_expect_tx(bar, STAGE_BYTES);
    tma_load_3d(st + ST_K0, tk, bar, 0, t0, bhk);
    tma_load_3d(st + ST_Q0, tq, bar, 0, t0, bhk);
    tma_load_3d(st + ST_K1, tk, bar, 64, t0, bhk);
    tma_load_3d(st + ST_Q1, tq, bar, 64, t0, bhk);
    tma_load_3d(st + ST_V0, tv, bar, 0, t0, bh);
    tma_load_3d(st + ST_V1, tv, bar, 64, t0, bh);
}

// T = (I + A)^-1 for a strictly lower 64x64 A (fp32, fidx layout), blocked in
// 16x16: diagonal blocks by forward substitution, then the off-diagonal
// blocks by block elimination  T_ij = -T_ii (sum_k A_ik T_kj)  in two levels.
__device__ __forceinline__ void solve_unit_lower_64(const float* A, float* T, int tid) {
    // Level 0: the four diagonal 16x16 blocks; the upper blocks are zeroed.
    if (tid < 64) {
        const int base = (tid >> 4) * 16, jj = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == jj) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) acc -= A[fidx(base + i, base + m)] * x[m];
            x[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) T[fidx(base + i, base + jj)] = x[i];
    } else {
        for (int e = tid - 64; e < 6 * 256; e += 64) {
            const int blk = e >> 8, w = e & 255;
            // upper blocks (bi, bj), bi < bj: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
            const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            T[fidx(bi * 16 + (w >> 4), bj * 16 + (w & 15))] = 0.f;
        }
    }
    __syncthreads();
    // Level 1: blocks (1,0), (2,1), (3,2).  96 threads: 16 rows x 2 column halves per block.
    float y[8];
    const bool l1 = tid < 96;
    const int blk = tid >> 5, r16 = tid & 15, c8 = ((tid >> 4) & 1) * 8;
    if (l1) {
        const int rb = 16 * (blk + 1), cb = 16 * blk;
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 4
        for (int m = 0; m < 16; ++m) {
            const float a = A[fidx(rb + r16, cb + m)];
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] += a * T[fidx(cb + m, cb + c8 + u)];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) T[fidx(rb + r16, cb + c8 + u)] = y[u];  // X = A_(b+1,b) T_bb
    }
    __syncthreads();
    if (l1) {
        const int rb = 16 * (blk + 1), cb = 16 * blk;
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 4
        for (int m = 0; m < 16; ++m) {
            const float t = T[fidx(rb + r16, rb + m)];
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] -= t * T[fidx(rb + m, cb + c8 + u)];
        }
    }
    __syncthreads();
    if (l1) {
        const int rb = 16 * (blk + 1), cb = 16 * blk;
#pragma unroll
        for (int u = 0; u < 8; ++u) T[fidx(rb + r16, cb + c8 + u)] = y[u];
    }
    __syncthreads();
    // Level 2: block rows 32..63 x cols 0..31.  Thread: row 32 + (tid & 31), 8 columns.
    const int r32 = tid & 31, c32 = (tid >> 5) * 8;
#pragma unroll
    for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 4
    for (int m = 0; m < 32; ++m) {
        const float a = A[fidx(32 + r32, m)];
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] += a * T[fidx(m, c32 + u)];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) T[fidx(32 + r32, c32 + u)] = y[u];
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) y[u] = 0.f;
#pragma unroll 4
    for (int m = 0; m < 32; ++m) {
        const float t = T[fidx(32 + r32, 32 + m)];
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] -= t * T[fidx(32 + m, c32 + u)];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) T[fidx(32 + r32, c32 + u)] = y[u];
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
    gdn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                          const float* __restrict__ g_log, const float* __restrict__ beta,
                          float* __restrict__ state, float scale, int Hk, int Hv, int S, int zero_init,
                          int32_t* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    Shared sh;
    sh.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    sh.sbase = smem_u32(sh.base);
    sh.G = reinterpret_cast<float*>(sh.base + OFF_SMALL);
    sh.gam = sh.G + 64;
    sh.bet = sh.G + 128;
    sh.ec = sh.G + 192;
    sh.bar_tma = reinterpret_cast<uint64_t*>(sh.base + OFF_BAR);
    sh.bar_mma = sh.bar_tma + 2;
    sh.tmem_slot = reinterpret_cast<uint32_t*>(sh.bar_mma + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int bh = blockIdx.x;
    const int b = bh / Hv;
    const int h = bh - b * Hv;
    const int bhk = b * Hk + h / (Hv / Hk);
    const int n_chunks = (S + kC - 1) / kC;

    float* As = reinterpret_cast<float*>(sh.base + OFF_OUT);  // fp32 A during the solve
    float* Ts = reinterpret_cast<float*>(sh.base + OFF_DT);   // fp32 T during the solve

    if (tid == 0) {
        mbar_init(&sh.bar_tma[0], 1);
        mbar_init(&sh.bar_tma[1], 1);
        mbar_init(sh.bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    if (warp == 0) {
        tmem_alloc(sh.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter

    // Loads issued so far (chunks [0, issued)); chunks whose loads were consumed: [0, consumed).
    int issued = 0, consumed = 0;
    uint32_t mma_phase = 0;
    bool mma_pending = false;
    bool failed = false;

    if (tid == 0) {
        for (; issued < 2 && issued < n_chunks; ++issued)
            issue_chunk_loads(sh, issued, &tm_q, &tm_k, &tm_v, issued * kC, bhk, bh);
    }

    // ---- initial state -> TMEM (S^T: lane dv, column dk) and its bf16 copy
    {
        const float* Sg = state + (size_t)bh * kD * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = zero_init ? 0.f : Sg[(size_t)(c0 + j) * kD + tid];
            tmem_st32(trow + COL_S + c0, r);
            st_row_bf16x32(sh.base + OFF_SB + (c0 >> 6) * 16384, tid, (c0 & 63) * 2, r);
        }
        tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
        const int stage = c & 1;
        const uint32_t st_s = sh.sbase + stage * STAGE_BYTES;
        const int t0 = c * kC;

        // (0) decay scan over the chunk (warps 0, 1: token r = tid)
        if (tid < 64) {
            const size_t gi = (size_t)bh * S + t0;
            const int ta = lane, tb = 32 + lane;
            float ga = (t0 + ta < S) ? g_log[gi + ta] : 0.f;
            float gb = (t0 + tb < S) ? g_log[gi + tb] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float ua = __shfl_up_sync(0xffffffffu, ga, o);
                const float ub = __shfl_up_sync(0xffffffffu, gb, o);
                if (lane >= o) {
                    ga += ua;
                    gb += ub;
                }
            }
            const float tot_a = __shfl_sync(0xffffffffu, ga, 31);
            gb += tot_a;
            const float gC = __shfl_sync(0xffffffffu, gb, 31);
            const float gr = warp == 0 ? ga : gb;
            const int r = tid;
            sh.G[r] = gr;
            sh.gam[r] = expf(gr);
            sh.bet[r] = (t0 + r < S) ? beta[gi + r] : 0.f;
            sh.ec[r] = expf(gC - gr);
        }

        // (1) chunk inputs landed -> [K;Q] K^T and S0^T Q^T
        failed = !mbar_wait(&sh.bar_tma[stage], (c >> 1) & 1);
        if (__syncthreads_or(failed)) goto abort;
        consumed = c + 1;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + COL_KQ, make_sdesc(st_s + ST_K0 + off, 16, 1024),
                         make_sdesc(st_s + ST_K0 + off, 16, 1024), IDESC_N64_KK, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + COL_QS, make_sdesc(sh.sbase + OFF_SB + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                         make_sdesc(st_s + ST_Q0 + off, 16, 1024), IDESC_N64_KK, kk > 0);
            }
            mma_commit(sh.bar_mma);
            tma_store_wait_read0();  // the previous out tile has left the staging area (A reuses it)
        }
        mma_pending = true;
        failed = !mbar_wait(sh.bar_mma, mma_phase);
        if (__syncthreads_or(failed)) goto abort;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // (2) A (fp32, lanes 0..63) and P (bf16, lanes 64..127) from the Gram rows
        {
            float x0[32], x1[32];
            tmem_ld32(trow + COL_KQ, x0);
            tmem_ld32(trow + COL_KQ + 32, x1);
            tmem_wait_ld();
            if (tid < 64) {
                const int r = tid;
                const float Gr = sh.G[r], br = sh.bet[r];
#pragma unroll
                for (int j = 0; j < 32; ++j) As[fidx(r, j)] = (j < r) ? br * expf(Gr - sh.G[j]) * x0[j] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    As[fidx(r, 32 + j)] = (32 + j < r) ? br * expf(Gr - sh.G[32 + j]) * x1[j] : 0.f;
            } else {
                const int r = tid - 64;
                const float Gr = sh.G[r];
#pragma unroll
                for (int j = 0; j < 32; ++j) x0[j] = (j <= r) ? expf(Gr - sh.G[j]) * x0[j] : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) x1[j] = (32 + j <= r) ? expf(Gr - sh.G[32 + j]) * x1[j] : 0.f;
                st_row_bf16x32(sh.base + OFF_P, r, 0, x0);
                st_row_bf16x32(sh.base + OFF_P, r, 64, x1);
            }
        }
        __syncthreads();

        // (3) T = (I + A)^-1 (fp32), then T diag(beta) and T diag(beta gamma) as bf16
        solve_unit_lower_64(As, Ts, tid);
        {
            const int r = tid >> 1, j0 = (tid & 1) * 32;
            float t1[32], t2[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float t = Ts[fidx(r, j0 + j)];
                const float bj = sh.bet[j0 + j];
                t1[j] = t * bj;
                t2[j] = t * bj * sh.gam[j0 + j];
            }
            st_row_bf16x32(sh.base + OFF_T1, r, j0 * 2, t1);
            st_row_bf16x32(sh.base + OFF_T2, r, j0 * 2, t2);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // (4) U^T = V^T T1^T,  W^T = K^T T2^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + COL_U, make_sdesc(st_s + ST_V0 + kk * 2048, 8192, 1024),
                         make_sdesc(sh.sbase + OFF_T1 + kk * 32, 16, 1024), IDESC_N64_MK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + COL_W, make_sdesc(st_s + ST_K0 + kk * 2048, 16384, 1024),
                         make_sdesc(sh.sbase + OFF_T2 + kk * 32, 16, 1024), IDESC_N64_MK, kk > 0);
            mma_commit(sh.bar_mma);
        }
        mma_pending = true;
        failed = !mbar_wait(sh.bar_mma, mma_phase);
        if (__syncthreads_or(failed)) goto abort;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // (5) -W as the MN-major B operand: row dk = tid, 64 token values
        {
            float x0[32], x1[32];
            tmem_ld32(trow + COL_W, x0);
            tmem_ld32(trow + COL_W + 32, x1);
            tmem_wait_ld();
            st_row_bf16x32(sh.base + OFF_WD, tid, 0, x0, -1.f);
            st_row_bf16x32(sh.base + OFF_WD, tid, 64, x1, -1.f);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // (6) Delta^T = U^T + S0^T (-W)^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + COL_U, make_sdesc(sh.sbase + OFF_SB + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                         make_sdesc(sh.sbase + OFF_WD + kk * 2048, 8192, 1024), IDESC_N64_KM, 1);
            mma_commit(sh.bar_mma);
        }
        mma_pending = true;
        failed = !mbar_wait(sh.bar_mma, mma_phase);
        if (__syncthreads_or(failed)) goto abort;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // (7) Delta^T and Delta~^T = Delta^T diag(exp(G_C - G)) as K-major A operands (row dv = tid)
        {
            float x0[32], x1[32];
            tmem_ld32(trow + COL_U, x0);
            tmem_ld32(trow + COL_U + 32, x1);
            tmem_wait_ld();
            st_row_bf16x32(sh.base + OFF_WD, tid, 0, x0);
            st_row_bf16x32(sh.base + OFF_WD, tid, 64, x1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x0[j] *= sh.ec[j];
                x1[j] *= sh.ec[32 + j];
            }
            st_row_bf16x32(sh.base + OFF_DT, tid, 0, x0);
            st_row_bf16x32(sh.base + OFF_DT, tid, 64, x1);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // (8) R_PD = Delta^T P^T,  R_SN = Delta~^T K
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + COL_KQ, make_sdesc(sh.sbase + OFF_WD + kk * 32, 16, 1024),
                         make_sdesc(sh.sbase + OFF_P + kk * 32, 16, 1024), IDESC_N64_KK, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + COL_SN, make_sdesc(sh.sbase + OFF_DT + kk * 32, 16, 1024),
                         make_sdesc(st_s + ST_K0 + kk * 2048, 16384, 1024), IDESC_N128_KM, kk > 0);
            mma_commit(sh.bar_mma);
        }
        mma_pending = true;
        failed = !mbar_wait(sh.bar_mma, mma_phase);
        if (__syncthreads_or(failed)) goto abort;
        mma_phase ^= 1;
        mma_pending = false;
        tc_fence_after();

        // (9) state S^T <- gamma_C S^T + R_SN (fp32 in TMEM) and its bf16 copy
        {
            const float gC = sh.gam[kC - 1];
#pragma unroll 1
            for (int c0 = 0; c0 < kD; c0 += 32) {
                float s[32], dn[32];
                tmem_ld32(trow + COL_S + c0, s);
                tmem_ld32(trow + COL_SN + c0, dn);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = fmaf(gC, s[j], dn[j]);
                tmem_st32(trow + COL_S + c0, s);
                st_row_bf16x32(sh.base + OFF_SB + (c0 >> 6) * 16384, tid, (c0 & 63) * 2, s);
            }
        }
        // (10) output O^T[dv][r] = scale (gamma_r R_QS + R_PD) -> bf16 tile [r][dv]
        {
            uint8_t* ob = sh.base + OFF_OUT + (tid >> 6) * 8192;
            const uint32_t cb = (uint32_t)(tid & 63) * 2;
#pragma unroll 1
            for (int r0 = 0; r0 < kC; r0 += 32) {
                float qs[32], pd[32];
                tmem_ld32(trow + COL_QS + r0, qs);
                tmem_ld32(trow + COL_KQ + r0, pd);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float o = scale * fmaf(sh.gam[r0 + j], qs[j], pd[j]);
                    *reinterpret_cast<__nv_bfloat16*>(ob + sw128_offset(r0 + j, cb)) = __float2bfloat16_rn(o);
                }
            }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&tm_o, sh.base + OFF_OUT, 0, t0, bh);
            tma_store_3d(&tm_o, sh.base + OFF_OUT + 8192, 64, t0, bh);
            tma_store_commit();
            if (issued < n_chunks) {  // this stage's tiles are no longer read by any MMA
                issue_chunk_loads(sh, stage, &tm_q, &tm_k, &tm_v, issued * kC, bhk, bh);
                ++issued;
            }
        }
    }

    // ---- final state S[dk][dv] = S^T[dv][dk] (coalesced across a warp)
    {
        tc_fence_after();
        float* Sg = state + (size_t)bh * kD * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
            float s[32];
            tmem_ld32(trow + COL_S + c0, s);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) Sg[(size_t)(c0 + j) * kD + tid] = s[j];
        }
    }
    if (tid == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    return;

abort:
    // A wait gave up: record it, drain what is still in flight (bounded), free TMEM.
    if (tid == 0) {
        atomicExch(status, (int32_t)GDN_ERR_TIMEOUT);
        for (int cc = consumed; cc < issued; ++cc) (void)mbar_wait(&sh.bar_tma[cc & 1], (cc >> 1) & 1);
        if (mma_pending) (void)mbar_wait(sh.bar_mma, mma_phase);
        tma_store_wait_all0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

// [heads, S, 128] bf16 viewed as a 3-D tensor (128 innermost), box 64 x 64 x 1.
bool encode_bf16_3d(CUtensorMap* map, const void* ptr, int heads, int S) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)S, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)S * kD * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const Problem& p) { return p.bf16 && p.Dk == kD && p.Dv == kD; }

gdn_status launch_prefill_tc(const Problem& p, int32_t* status_word, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    if (!encode_bf16_3d(&tq, p.q, p.B * p.Hk, p.S) || !encode_bf16_3d(&tk, p.k, p.B * p.Hk, p.S) ||
        !encode_bf16_3d(&tv, p.v, p.B * p.Hv, p.S) || !encode_bf16_3d(&to, p.out, p.B * p.Hv, p.S))
        return GDN_ERR_CUDA;
    if (cudaFuncSetAttribute(gdn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_ALLOC) != cudaSuccess)
        return GDN_ERR_CUDA;
    gdn_prefill_tc_kernel<<<p.B * p.Hv, kThreads, SMEM_ALLOC, stream>>>(
        tq, tk, tv, to, p.g_log, p.beta, p.state, p.scale, p.Hk, p.Hv, p.S, p.zero_init ? 1 : 0, status_word);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
