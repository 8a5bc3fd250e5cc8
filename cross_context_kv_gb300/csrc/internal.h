// internal.h -- declarations shared by the host-side translation units of libkvfix.
// Not part of the public ABI (include/kvfix.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvfix.h"

namespace kvfix {

// Host-computed RoPE frequencies theta_i = base^(-2i/D), passed by value to kernels.
constexpr int kMaxHeadDim = 256;
struct RopeTheta {
    double theta[kMaxHeadDim / 2];
};
RopeTheta make_theta(double base, int head_dim);

// Records `msg` as the calling thread's last error and returns `st`.
kvfix_status fail(kvfix_status st, const char* fmt, ...);
// Maps a CUDA error (after a launch or runtime call) to KVFIX_ECUDA with a message.
kvfix_status cuda_fail(cudaError_t err, const char* what);

// Per-translation-unit device status words: read (and clear) on `stream`.
unsigned read_status_repair(cudaStream_t stream);
unsigned read_status_diff(cudaStream_t stream);
unsigned read_status_draft(cudaStream_t stream);
unsigned read_status_lowrank(cudaStream_t stream);
unsigned read_status_lowrank_draft(cudaStream_t stream);

// ---- launchers (enqueue only; arguments already validated) -----------------------

cudaError_t launch_rerope(const uint16_t* in, const kvfix_kv_desc& d, uint16_t* out,
                          const kvfix_kv_desc& od, const int32_t* delta, const RopeTheta& th,
                          cudaStream_t s);

cudaError_t launch_score(const uint16_t* k_reuse, const uint16_t* v_reuse,
                         const kvfix_kv_desc& reuse, const uint16_t* k_fresh,
                         const uint16_t* v_fresh, const kvfix_kv_desc& fresh, int agents,
                         const int32_t* delta, const RopeTheta& th, float* d_k, float* d_v,
                         float* w_k, float* w_v, uint32_t* mask_union, cudaStream_t s);

// Top-b of float scores per unit for two planes (either may be skipped with NULL
// scores), plus the optional union mask.
cudaError_t launch_select_f32(const float* d_k, const float* d_v, int units, int n, int b,
                              int32_t* idx_k, int32_t* idx_v, uint32_t* mask_k,
                              uint32_t* mask_v, uint32_t* mask_union, cudaStream_t s);

// Both planes of one kvfix_mean_correct call (index 0 = K, rotated; 1 = V); a plane
// whose reuse pointer is null is skipped.
struct McPlanes {
    const uint16_t* reuse[2];
    const uint16_t* fresh[2];
    uint16_t* out[2];
    const int32_t* idx[2];
    const float* w[2];
    float* mu[2];
};
cudaError_t launch_mean_correct(const McPlanes& planes, const kvfix_kv_desc& rd,
                                const kvfix_kv_desc& fd, const kvfix_kv_desc& od, int agents,
                                const int32_t* delta, const RopeTheta& th, int b, cudaStream_t s);

cudaError_t launch_lowrank(const uint16_t* x, const kvfix_kv_desc& d, const uint16_t* A,
                           const uint16_t* B, int rank, uint16_t* out, const kvfix_kv_desc& od,
                           cudaStream_t s);

size_t draft_workspace_bytes(const kvfix_kv_desc& d, int layer_begin);
cudaError_t launch_draft(const uint16_t* k, const kvfix_kv_desc& d, const uint16_t* q,
                         int steps, int q_heads, int layer_begin, int k_rows, int32_t* idx,
                         double* scores, void* ws, cudaStream_t s);
// The draft-rank tail shared by the fused low-rank call: the per-key masses of each
// chunk's units (contrib [chunks][units_per_chunk][n]) summed into scores, then the top
// k_rows of each chunk.
cudaError_t launch_draft_finish(const float* contrib, int chunks, int n, long long units_per_chunk, int k_rows,
                                int32_t* idx, double* scores, cudaStream_t s);
// Low-rank delta of the key plane fused with the draft scoring of the corrected keys:
// out = x + A B (every layer), and for layers >= layer_begin the per-key attention
// masses of the draft queries into contrib (as launch_draft's first stage); then the
// draft-rank tail.
size_t lowrank_draft_workspace_bytes(const kvfix_kv_desc& d, int layer_begin);
cudaError_t launch_lowrank_draft(const uint16_t* x, const kvfix_kv_desc& d, const uint16_t* A, const uint16_t* B,
                                 int rank, uint16_t* out, const kvfix_kv_desc& od, const uint16_t* q, int steps,
                                 int q_heads, int layer_begin, int k_rows, int32_t* idx, double* scores, void* ws,
                                 cudaStream_t s);
// Rows idx[c][0 .. k_rows) (or the first counts[c] of them, counts non-null) of io are
// overwritten with the same rows of fresh, every layer and head.
cudaError_t launch_row_repair(uint16_t* io, const kvfix_kv_desc& d, const uint16_t* fresh,
                              const kvfix_kv_desc& fd, const int32_t* idx, int k_rows,
                              cudaStream_t s, const int32_t* counts = nullptr);

// Repair layouts: one CTA per unit (tokens <= 16384).
unsigned read_status_layout(cudaStream_t stream);
size_t layout_smem_bytes(int n, int layout, int B, int k);
cudaError_t launch_repair_layout(const double* scores, int units, int n, int layout, int B, int k, int c,
                                 int skipped, double tau, int32_t* idx, int max_rows, int32_t* counts,
                                 cudaStream_t s);

// mask_v non-null: K blocks are marked in mask and V blocks in mask_v (per-plane lists).
cudaError_t launch_diff_mask(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                             const uint16_t* sk, const uint16_t* sv, const kvfix_kv_desc& sd,
                             int bt, uint32_t* mask, cudaStream_t s, uint32_t* mask_v = nullptr);
cudaError_t launch_diff_scan(const uint32_t* mask, int siblings, long long per_sibling,
                             int64_t* offsets, cudaStream_t s);
// planes: 0 = entries hold the K block then the V block; 1 = K only; 2 = V only.
cudaError_t launch_diff_pack(const uint16_t* sk, const uint16_t* sv, const kvfix_kv_desc& sd,
                             int bt, const uint32_t* mask, const int64_t* offsets,
                             uint16_t* payload, long long capacity, cudaStream_t s, int planes = 0);
cudaError_t launch_diff_gather(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                               const uint32_t* mask, const int64_t* offsets,
                               const uint16_t* payload, long long payload_entries, int siblings,
                               int bt, uint16_t* ok, uint16_t* ov, const kvfix_kv_desc& od,
                               cudaStream_t s, const uint32_t* mask_v = nullptr,
                               const int64_t* offsets_v = nullptr, const uint16_t* payload_v = nullptr,
                               long long entries_v = 0);
// Per-agent total deviation (double) and the agent with the smallest one.
cudaError_t launch_master_select(const float* d_k, const float* d_v, int agents, int units_per_agent,
                                 int tokens, double* totals, int32_t* master, cudaStream_t s);

cudaError_t launch_diff_restore(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                                const uint32_t* mask, const int64_t* offsets,
                                const uint16_t* payload, long long payload_entries, int siblings,
                                int bt, const int32_t* delta, const RopeTheta& th,
                                const int32_t* slot_map, uint16_t* pk, uint16_t* pv,
                                const kvfix_kv_desc& pd, cudaStream_t s, const uint32_t* mask_v = nullptr,
                                const int64_t* offsets_v = nullptr, const uint16_t* payload_v = nullptr,
                                long long entries_v = 0);

// Anchor-pool correction (both planes: index 0 = keys, rotated; 1 = values).
struct AnchorPlanes {
    const uint16_t* src[2];
    const uint16_t* ac[2];
    const uint16_t* bct[2];
    const uint16_t* ad[2];
    const uint16_t* bdt[2];
    float* w[2];
    uint16_t* out[2];
};
unsigned read_status_anchor(cudaStream_t stream);
bool anchor_shape_ok(int anchors, int rank, int head_dim);
size_t anchor_gate_workspace_bytes(const kvfix_kv_desc& d, int anchors, int prefix);
cudaError_t launch_anchor_gate(const uint16_t* v_src, const kvfix_kv_desc& d, const uint16_t* ac,
                               const uint16_t* bct, int V, int r, int k, double T, double tau,
                               double* dist, double* g, double* hbar, int32_t* accept,
                               void* workspace, cudaStream_t s);
// With gate non-null, the gate is computed in the same pass (value plane, prefix k) and
// its accept flags decide which segments are corrected.
struct AnchorGateOut {
    int k;
    double T, tau;
    double* d;
    double* g;
    double* hbar;
    int32_t* accept;
    void* workspace;  // anchor_gate_workspace_bytes(d, V, tokens)
};
cudaError_t launch_anchor_correct(const AnchorPlanes& pl, const kvfix_kv_desc& d,
                                  const kvfix_kv_desc& od, int V, int r, double T,
                                  const int32_t* delta, const RopeTheta& th, const int32_t* accept,
                                  cudaStream_t s, const AnchorGateOut* gate = nullptr);

// Bounded-wait self test.
unsigned read_status_selftest(cudaStream_t stream);
cudaError_t launch_selftest_wait(long long limit_cycles, const int* flag, cudaStream_t s);

}  // namespace kvfix
