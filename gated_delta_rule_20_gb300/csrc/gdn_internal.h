// gdn_internal.h -- declarations shared by the host entry points and the
// kernel launchers of the GDN library (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {

// One call's arguments after host-side validation.
struct Problem {
    const void* q;
    const void* k;
    const void* v;
    const float* g_log;
    const float* beta;
    float scale;
    float* state;  // in/out, [B, Hv, Dk, Dv]
    void* out;
    int B, Hk, Hv, S, Dk, Dv;
    bool bf16;       // compute dtype of q/k/v/out
    bool zero_init;  // GDN_ZERO_INITIAL_STATE
    bool single_pass = false;  // GDN_SINGLE_PASS: never split a sequence into segments
};

// Device address of the current device's kernel-side status word (0 = fine,
// else a gdn_status written by a kernel whose wait gave up).
gdn_status status_word_for_current_device(int32_t** out);

// The argument checks of gdn_prefill, without launching anything.
gdn_status prefill_checked(const void* q, const void* k, const void* v, const float* g_log, const float* beta,
                           float* state, void* out, const gdn_dims* d);

// Decode step (S == 1): one pass over the fp32 state.
cudaError_t launch_decode(const Problem& p, cudaStream_t stream);

// Chunked prefill on FP32 FFMA (any supported dims, fp32 or bf16 inputs).
cudaError_t launch_prefill_ffma(const Problem& p, cudaStream_t stream);

// Chunked prefill on tcgen05 tensor cores (bf16, Dk = Dv = 128).
bool prefill_tc_supported(const Problem& p);
// Segments the tensor-core prefill splits each sequence into on a device with `sms` SMs
// (1: one pass).
int prefill_tc_segments(const Problem& p, int sms);
// The same, and with capacity >= P + 1 the segments' first tokens in starts[0 .. P - 1] and
// S in starts[P].
int prefill_tc_segment_starts(const Problem& p, int sms, long long* starts, int capacity);
// Device scratch of launch_prefill_tc on a device with `sms` SMs: the segment states, maps
// and the identity-start runs' outputs of a split (0 for one pass).
size_t prefill_tc_workspace_bytes(const Problem& p, int sms);
// workspace == nullptr: a split takes stream-ordered scratch itself (and runs one pass if it
// cannot be had); otherwise the caller's buffer of workspace_bytes >=
// prefill_tc_workspace_bytes(p, SM count) bytes, 16-byte aligned, is used.
gdn_status launch_prefill_tc(const Problem& p, int* status_word, cudaStream_t stream, void* workspace,
                             size_t workspace_bytes);
// The tensor-core prefill's wait limit on the current device (0: the default second).
cudaError_t set_prefill_tc_wait_limit(unsigned long long ns);
// The tensor-core prefill's test hook on the current device (see gdn_test_stall_prefill).
cudaError_t set_prefill_tc_test_stall(int on);

// The conv1d decode step folded into the gated step: q|k|v are computed from the
// already shifted windows [B, conv_dim, K] bf16 (the newest token last) and the
// taps [conv_dim, K] fp32 instead of being read.
struct GatedConvInput {
    const void* window;
    const float* weight;
    int K;
};

// gdn_decode_gated after its argument checks (qkv unused when conv is given;
// conv requires bf16).  With after_producer the kernel is launched with
// programmatic stream serialization: it may start while the preceding kernel of
// the stream runs (that kernel must execute griddepcontrol.launch_dependents),
// and reads nothing but the state before that kernel has completed.  next_head,
// when not null, is a device counter that is zero once the preceding kernel has
// completed: the streaming kernel then hands out heads dynamically.
gdn_status decode_gated_checked(const void* qkv, const void* z, const void* a, const void* b, const float* A_log,
                                const float* dt_bias, const float* norm_weight, float scale, float* state_inout,
                                void* out, const gdn_dims* d, cudaStream_t stream, bool after_producer,
                                const GatedConvInput* conv, int* next_head);

}  // namespace gdn
