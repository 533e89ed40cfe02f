// gdn_api.cu -- the library's extern "C" entry points: host-side argument
// checks, dispatch to the kernels, and the per-device kernel status word.
//
// Argument rules follow the "GDN CTE Kernel API Reference" page (Parameters,
// Notes, Dimensions): Dq == Dk <= 128, Dv <= 128, Hv % Hk == 0, fp32 g_log /
// beta / state, compute dtype from the query.  A failed check launches nothing.
#include <cstdint>
#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {
// Kernel-side status word of each device (0 = fine, else a gdn_status).  Its
// device address is looked up once per device, with that device current.
__device__ int32_t g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_status_addr[kMaxDevices] = {};

}  // namespace

gdn_status status_word_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return GDN_ERR_CUDA;
        g_status_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_status_addr[dev];
    return GDN_OK;
}


namespace {

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

constexpr uint32_t kKnownFlags = GDN_ZERO_INITIAL_STATE | GDN_FORCE_FFMA | GDN_SINGLE_PASS;

gdn_status check(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                 float* state, void* out, const gdn_dims* d, bool decode, Problem* p) {
    if (!d) return GDN_ERR_NULL;
    if (d->dtype != GDN_F32 && d->dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (d->flags & ~kKnownFlags) return GDN_ERR_UNSUPPORTED;
    if (d->B < 0 || d->Hk < 1 || d->Hv < 1 || d->S < 0 || d->Dk < 1 || d->Dv < 1) return GDN_ERR_DIMS;
    if (d->Dk > 128 || d->Dv > 128) return GDN_ERR_DIMS;  // MAX_HEAD_DIM (Notes)
    if (d->Hv % d->Hk != 0) return GDN_ERR_DIMS;          // GQA (Notes)
    if (decode && d->S != 1) return GDN_ERR_DIMS;
    // Index arithmetic inside the kernels uses 32-bit (b, head, token) counters.
    if (d->B * d->Hv > INT32_MAX || d->S > INT32_MAX || d->B > INT32_MAX) return GDN_ERR_DIMS;
    const bool empty = d->B == 0 || d->S == 0;
    if (!state) return GDN_ERR_NULL;
    if (!empty && (!q || !k || !v || !g_log || !beta || !out)) return GDN_ERR_NULL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(g_log) || misaligned(beta) ||
        misaligned(state) || misaligned(out))
        return GDN_ERR_ALIGN;
    p->q = q;
    p->k = k;
    p->v = v;
    p->g_log = g_log;
    p->beta = beta;
    p->state = state;
    p->out = out;
    p->B = (int)d->B;
    p->Hk = (int)d->Hk;
    p->Hv = (int)d->Hv;
    p->S = (int)d->S;
    p->Dk = (int)d->Dk;
    p->Dv = (int)d->Dv;
    p->bf16 = d->dtype == GDN_BF16;
    p->zero_init = (d->flags & GDN_ZERO_INITIAL_STATE) != 0;
    p->single_pass = (d->flags & GDN_SINGLE_PASS) != 0;
    return GDN_OK;
}

// S == 0: no tokens; the final state equals the initial one (zero under
// GDN_ZERO_INITIAL_STATE).
gdn_status empty_sequence(const Problem& p, cudaStream_t stream) {
    if (p.B == 0 || !p.zero_init) return GDN_OK;
    const size_t bytes = (size_t)p.B * p.Hv * p.Dk * p.Dv * sizeof(float);
    return cudaMemsetAsync(p.state, 0, bytes, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

gdn_status prefill_checked(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                           float* state, void* out, const gdn_dims* d) {
    Problem p{};
    return check(q, k, v, g_log, beta, state, out, d, false, &p);
}

}  // namespace gdn

extern "C" {

gdn_status gdn_prefill_ws(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                          float scale, float* state_inout, void* out, const gdn_dims* dims, void* workspace,
                          size_t workspace_bytes, gdn_stream_t stream) {
    gdn::Problem p{};
    p.scale = scale;
    gdn_status s = gdn::check(q, k, v, g_log, beta, state_inout, out, dims, false, &p);
    if (s != GDN_OK) return s;
    if (workspace && gdn::misaligned(workspace)) return GDN_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (p.B == 0 || p.S == 0) return gdn::empty_sequence(p, st);
    if (!(dims->flags & GDN_FORCE_FFMA) && gdn::prefill_tc_supported(p)) {
        int32_t* status = nullptr;
        s = gdn::status_word_for_current_device(&status);
        if (s != GDN_OK) return s;
        return gdn::launch_prefill_tc(p, status, st, workspace, workspace_bytes);
    }
    return gdn::launch_prefill_ffma(p, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_prefill(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                       float scale, float* state_inout, void* out, const gdn_dims* dims, gdn_stream_t stream) {
    return gdn_prefill_ws(q, k, v, g_log, beta, scale, state_inout, out, dims, nullptr, 0, stream);
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                           float scale, float* state_inout, void* out, const gdn_dims* dims,
                           gdn_stream_t stream) {
    gdn::Problem p{};
    p.scale = scale;
    gdn_status s = gdn::check(q, k, v, g_log, beta, state_inout, out, dims, true, &p);
    if (s != GDN_OK) return s;
    if (p.B == 0) return GDN_OK;
    return gdn::launch_decode(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int32_t gdn_prefill_segment_starts(const gdn_dims* d, int32_t sm_count, int64_t* starts, int32_t capacity) {
    if (!d || sm_count < 1) return 0;
    if ((d->dtype != GDN_F32 && d->dtype != GDN_BF16) || (d->flags & ~gdn::kKnownFlags)) return 0;
    if (d->B < 0 || d->Hk < 1 || d->Hv < 1 || d->S < 0 || d->Dk < 1 || d->Dv < 1 || d->Dk > 128 || d->Dv > 128 ||
        d->Hv % d->Hk != 0 || d->B * d->Hv > INT32_MAX || d->S > INT32_MAX)
        return 0;
    gdn::Problem p{};
    p.B = (int)d->B;
    p.Hk = (int)d->Hk;
    p.Hv = (int)d->Hv;
    p.S = (int)d->S;
    p.Dk = (int)d->Dk;
    p.Dv = (int)d->Dv;
    p.bf16 = d->dtype == GDN_BF16;
    p.single_pass = (d->flags & GDN_SINGLE_PASS) != 0;
    if ((d->flags & GDN_FORCE_FFMA) || !gdn::prefill_tc_supported(p)) p.single_pass = true;
    long long buf[17];
    const int P = gdn::prefill_tc_segment_starts(p, sm_count, buf, 17);
    if (starts && capacity >= P + 1)
        for (int j = 0; j <= P; ++j) starts[j] = P > 1 ? buf[j] : (j == 0 ? 0 : d->S);
    return P;
}

int32_t gdn_prefill_segments(const gdn_dims* d, int32_t sm_count) {
    return gdn_prefill_segment_starts(d, sm_count, nullptr, 0);
}

size_t gdn_prefill_workspace_bytes(const gdn_dims* dims) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (gdn_prefill_segments(dims, sms) <= 1) return 0;  // also 0 for invalid dims
    gdn::Problem p{};
    p.B = (int)dims->B;
    p.Hk = (int)dims->Hk;
    p.Hv = (int)dims->Hv;
    p.S = (int)dims->S;
    p.Dk = (int)dims->Dk;
    p.Dv = (int)dims->Dv;
    p.bf16 = dims->dtype == GDN_BF16;
    p.single_pass = (dims->flags & GDN_SINGLE_PASS) != 0;
    return gdn::prefill_tc_workspace_bytes(p, sms);
}

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK: success";
        case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
        case GDN_ERR_DIMS: return "GDN_ERR_DIMS: dims violate B,S>=0, Hk,Hv>=1, Hv%Hk==0, 1<=Dk,Dv<=128 (decode: S==1)";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: dtype or flags not supported by this build";
        case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: a tensor pointer is not 16-byte aligned";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a kernel wait ran past its bound";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: the workspace is smaller than gdn_prefill_workspace_bytes";
    }
    return "unknown gdn_status";
}

gdn_status gdn_device_status(int device, int clear, int32_t* code) {
    if (!code) return GDN_ERR_NULL;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status s = GDN_OK;
    int32_t val = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&val, gdn::g_status_word, sizeof(val)) != cudaSuccess) {
        s = GDN_ERR_CUDA;
    } else if (clear) {
        const int32_t zero = 0;
        if (cudaMemcpyToSymbol(gdn::g_status_word, &zero, sizeof(zero)) != cudaSuccess) s = GDN_ERR_CUDA;
    }
    cudaSetDevice(prev);
    *code = val;
    return s;
}

gdn_status gdn_set_wait_limit_ns(int device, uint64_t ns) {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status s = GDN_OK;
    if (cudaDeviceSynchronize() != cudaSuccess || gdn::set_prefill_tc_wait_limit(ns) != cudaSuccess) s = GDN_ERR_CUDA;
    cudaSetDevice(prev);
    return s;
}

gdn_status gdn_test_stall_prefill(int device, int on) {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return GDN_ERR_CUDA;
    gdn_status s = GDN_OK;
    if (cudaDeviceSynchronize() != cudaSuccess || gdn::set_prefill_tc_test_stall(on) != cudaSuccess) s = GDN_ERR_CUDA;
    cudaSetDevice(prev);
    return s;
}

int gdn_kernels_per_call(void) { return 1; }

}  // extern "C"
