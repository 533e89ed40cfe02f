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
};

// Device address of the current device's kernel-side status word (0 = fine,
// else a gdn_status written by a kernel whose wait gave up).
gdn_status status_word_for_current_device(int32_t** out);

// Decode step (S == 1): one pass over the fp32 state.
cudaError_t launch_decode(const Problem& p, cudaStream_t stream);

// Chunked prefill on FP32 FFMA (any supported dims, fp32 or bf16 inputs).
cudaError_t launch_prefill_ffma(const Problem& p, cudaStream_t stream);

// Chunked prefill on tcgen05 tensor cores (bf16, Dk = Dv = 128).
bool prefill_tc_supported(const Problem& p);
gdn_status launch_prefill_tc(const Problem& p, int* status_word, cudaStream_t stream);

}  // namespace gdn
