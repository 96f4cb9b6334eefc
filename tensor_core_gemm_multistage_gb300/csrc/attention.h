// attention.h - internal interface between the C-ABI layer (gsr_api.cu) and the attention
// forward kernel (attention_fwd.cu).  Not installed; not part of the ABI.
#pragma once

#include "kernels.h"

namespace gsr {

struct AttnParams {
    int BH;                 // batch * heads
    int Sq, Skv;
    int causal;             // keep key k for query q when k <= q + causal_offset
    int causal_offset;      // Skv - Sq
    float scale_log2;       // softmax scale * log2(e)
    int head_group;         // item order: query blocks longest first within groups of this many heads
    int num_items;          // ceil(Sq / 256) * BH work items (two 128-query tiles of one head each)
    int* work;              // [0] the launch's next work item, [1] CTAs done taking items; 0 between launches
    __half* O;              // (BH, Sq, D) row-major
    float* lse;             // optional (BH, Sq): natural-log log-sum-exp of the scaled scores
    int* err;
    uint64_t timeout_ns;
    uint32_t test_flags;
};

// Attention forward: Q, K, V as 3-D tensor maps {D, seq, BH} with 64 x 128 x 1 boxes; a
// persistent grid of `grid` CTAs (one per SM at most) takes the p.num_items work items.
cudaError_t launch_attention(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const AttnParams& p, int D, int grid, cudaStream_t stream);
// O = 0, lse = -inf for `rows` rows of width D (no keys).
cudaError_t launch_attention_empty(__half* O, float* lse, long long rows, int D, cudaStream_t stream);

}  // namespace gsr
