// softmax.cuh -- softmax statistics of the draft-query logits, shared by kvfix_draft_rank
// and kvfix_lowrank_draft so that both compute the per-key masses with the same
// arithmetic in the same order (Budgeted Cache Repair, section 3: the row score is the
// softmax attention mass of the draft queries).
//
// Logits are in base-2 units (z = q.k / sqrt(D) * log2 e), so every term is one exp2f.
// Per query row a thread keeps the running maximum m of the logits it has seen and the sum
// s of exp2(z - m), rescaled whenever the maximum grows.  Partial (m, s) pairs are brought
// to a common maximum M with rescaled(), which gives 0 for a part that saw no logit.
#pragma once

#include <math.h>

namespace kvfix {

// Branch-free: with M = max(m, z) one of the two exponents is 0 and its exp2f exactly 1,
// so this is s * 2^(m - z) + 1 when z > m and s + 2^(z - m) otherwise (the first logit:
// m = -inf, s = 0 gives s = 1).
__device__ __forceinline__ void online_add(float& m, float& s, float z) {
    const float M = fmaxf(m, z);
    s = s * exp2f(m - M) + exp2f(z - M);
    m = M;
}

__device__ __forceinline__ float rescaled(float m, float s, float M) { return m == -INFINITY ? 0.f : s * exp2f(m - M); }

// The warp's (m, s) of one row: the maximum over the lanes, then the lanes' rescaled sums
// added by an xor tree (every lane ends with the same pair).
__device__ __forceinline__ void warp_combine(float& m, float& s) {
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float t = rescaled(m, s, M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    m = M;
    s = t;
}

// Four warps' pairs, added in the order given.
__device__ __forceinline__ void combine4(const float* m4, const float* s4, float& M, float& S) {
    M = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    S = ((rescaled(m4[0], s4[0], M) + rescaled(m4[1], s4[1], M)) + rescaled(m4[2], s4[2], M)) +
        rescaled(m4[3], s4[3], M);
}

}  // namespace kvfix
