// api.cu -- the C ABI of libkvfix: argument checks, error reporting, launches.
// Every public call validates its arguments on the host, returns KVFIX_EINVAL with a
// message before anything is enqueued, and otherwise enqueues kernels on `stream`.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "internal.h"

namespace kvfix {

static thread_local char g_last_error[512] = "";

kvfix_status fail(kvfix_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kvfix_status cuda_fail(cudaError_t err, const char* what) {
    return fail(KVFIX_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

RopeTheta make_theta(double base, int head_dim) {
    RopeTheta t;
    memset(&t, 0, sizeof t);
    for (int i = 0; i < head_dim / 2; ++i) t.theta[i] = pow(base, -2.0 * (double)i / (double)head_dim);
    return t;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Checks one plane descriptor and its pointer.  `what` names the argument.
static kvfix_status check_plane(const void* ptr, const kvfix_kv_desc& d, const char* what,
                                bool allow_null = false) {
    if (ptr == nullptr && !allow_null) return fail(KVFIX_EINVAL, "%s: null pointer", what);
    if (d.chunks < 0 || d.layers < 0 || d.tokens < 0)
        return fail(KVFIX_EINVAL, "%s: negative chunks/layers/tokens", what);
    if (d.kv_heads < 1 || d.head_dim < 16 || d.head_dim > kMaxHeadDim || d.head_dim % 16 != 0)
        return fail(KVFIX_EINVAL, "%s: kv_heads must be >= 1 and head_dim a multiple of 16 in [16, %d] (got %d heads x %d)",
                    what, kMaxHeadDim, d.kv_heads, d.head_dim);
    if (d.stride_chunk < 0 || d.stride_layer < 0 || d.stride_token < 0)
        return fail(KVFIX_EINVAL, "%s: negative stride", what);
    if (d.stride_chunk % 8 || d.stride_layer % 8 || d.stride_token % 8)
        return fail(KVFIX_EINVAL, "%s: strides must be multiples of 8 elements (16 bytes)", what);
    const long long row = (long long)d.kv_heads * d.head_dim;
    if (d.tokens > 1 && d.stride_token < row)
        return fail(KVFIX_EINVAL, "%s: stride_token %lld is smaller than a token row (%lld)", what,
                    (long long)d.stride_token, row);
    if (ptr && !aligned16(ptr)) return fail(KVFIX_EINVAL, "%s: pointer not 16-byte aligned", what);
    return KVFIX_OK;
}

static bool same_shape(const kvfix_kv_desc& a, const kvfix_kv_desc& b) {
    return a.layers == b.layers && a.tokens == b.tokens && a.kv_heads == b.kv_heads &&
           a.head_dim == b.head_dim;
}

// Byte extent [lo, hi) touched by a plane view.
static void extent(const void* p, const kvfix_kv_desc& d, uintptr_t* lo, uintptr_t* hi) {
    const long long row = (long long)d.kv_heads * d.head_dim;
    long long last = 0;
    if (d.chunks > 0 && d.layers > 0 && d.tokens > 0)
        last = (long long)(d.chunks - 1) * d.stride_chunk + (long long)(d.layers - 1) * d.stride_layer +
               (long long)(d.tokens - 1) * d.stride_token + row;
    *lo = (uintptr_t)p;
    *hi = (uintptr_t)p + 2 * (uintptr_t)last;
}

static bool overlaps(const void* a, const kvfix_kv_desc& da, const void* b, const kvfix_kv_desc& db) {
    if (!a || !b) return false;
    uintptr_t a0, a1, b0, b1;
    extent(a, da, &a0, &a1);
    extent(b, db, &b0, &b1);
    return a0 < b1 && b0 < a1;
}

static bool overlaps_bytes(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

static kvfix_status launched(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return cuda_fail(e, what);
    return KVFIX_OK;
}

}  // namespace kvfix

using namespace kvfix;

extern "C" {

int kvfix_version(void) { return 100; }

const char* kvfix_last_error(void) { return g_last_error; }

kvfix_status kvfix_check_status(void* stream) {
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "kvfix_check_status: stream synchronize");
    unsigned bits = read_status_repair(s) | read_status_diff(s) | read_status_draft(s) | read_status_lowrank(s) |
                    read_status_anchor(s) | read_status_layout(s) | read_status_selftest(s) |
                    read_status_lowrank_draft(s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kvfix_check_status: status read");
    if (bits & 8u) return fail(KVFIX_EDEVICE, "a kernel's shared-memory layout check failed; its work was skipped");
    if (bits & 4u) return fail(KVFIX_ETIMEOUT, "a bounded device wait gave up");
    if (bits & 2u) return fail(KVFIX_ENOSPACE, "diff payload entries beyond the capacity were skipped");
    if (bits & 1u) return fail(KVFIX_EDEVICE, "an index in caller data was out of range and skipped");
    g_last_error[0] = '\0';
    return KVFIX_OK;
}

static bool same_desc(const kvfix_kv_desc& a, const kvfix_kv_desc& b) {
    return memcmp(&a, &b, sizeof a) == 0;
}

kvfix_status kvfix_rerope(const kvfix_bf16* k_in, kvfix_kv_desc in_desc, kvfix_bf16* k_out,
                          kvfix_kv_desc out_desc, const int32_t* delta, double rope_base,
                          void* stream) {
    kvfix_status st;
    if ((st = check_plane(k_in, in_desc, "kvfix_rerope: k_in")) != KVFIX_OK) return st;
    if ((st = check_plane(k_out, out_desc, "kvfix_rerope: k_out")) != KVFIX_OK) return st;
    if (!same_shape(in_desc, out_desc) || in_desc.chunks != out_desc.chunks)
        return fail(KVFIX_EINVAL, "kvfix_rerope: k_in and k_out shapes differ");
    if (in_desc.chunks > 0 && delta == nullptr) return fail(KVFIX_EINVAL, "kvfix_rerope: delta is null");
    if (!(rope_base > 1.0) || !isfinite(rope_base))
        return fail(KVFIX_EINVAL, "kvfix_rerope: rope_base must be finite and > 1");
    const bool in_place = (const void*)k_in == (const void*)k_out && same_desc(in_desc, out_desc);
    if (!in_place && overlaps(k_in, in_desc, k_out, out_desc))
        return fail(KVFIX_EINVAL, "kvfix_rerope: k_out overlaps k_in (only an exact in-place call is allowed)");
    RopeTheta th = make_theta(rope_base, in_desc.head_dim);
    return launched(launch_rerope(k_in, in_desc, k_out, out_desc, delta, th, (cudaStream_t)stream),
                    "kvfix_rerope");
}

kvfix_status kvfix_score_topk(const kvfix_bf16* k_reuse, const kvfix_bf16* v_reuse,
                              kvfix_kv_desc reuse, const kvfix_bf16* k_fresh,
                              const kvfix_bf16* v_fresh, kvfix_kv_desc fresh, int32_t agents,
                              const int32_t* delta, double rope_base, int32_t b, float* d_k,
                              float* d_v, float* w_k, float* w_v, int32_t* idx_k, int32_t* idx_v,
                              uint32_t* mask_k, uint32_t* mask_v, uint32_t* mask_union,
                              void* stream) {
    kvfix_status st;
    const char* fn = "kvfix_score_topk";
    if ((st = check_plane(k_reuse, reuse, "kvfix_score_topk: k_reuse")) != KVFIX_OK) return st;
    if ((st = check_plane(v_reuse, reuse, "kvfix_score_topk: v_reuse")) != KVFIX_OK) return st;
    if ((st = check_plane(k_fresh, fresh, "kvfix_score_topk: k_fresh")) != KVFIX_OK) return st;
    if ((st = check_plane(v_fresh, fresh, "kvfix_score_topk: v_fresh")) != KVFIX_OK) return st;
    if (reuse.layers != 1 || fresh.layers != 1)
        return fail(KVFIX_EINVAL, "%s: reuse and fresh must be check-layer views (layers == 1)", fn);
    if (!same_shape(reuse, fresh)) return fail(KVFIX_EINVAL, "%s: reuse and fresh shapes differ", fn);
    if (agents < 1) return fail(KVFIX_EINVAL, "%s: agents must be >= 1", fn);
    const long long units = (long long)agents * reuse.chunks;
    if (fresh.chunks != units)
        return fail(KVFIX_EINVAL, "%s: fresh.chunks (%d) must equal agents*reuse.chunks (%lld)", fn,
                    fresh.chunks, units);
    if (units > 65535 || reuse.chunks > 65535) return fail(KVFIX_EINVAL, "%s: at most 65535 units", fn);
    const int n = reuse.tokens;
    if (n > 65536) return fail(KVFIX_EINVAL, "%s: tokens must be <= 65536", fn);
    if (b < 0 || b > n) return fail(KVFIX_EINVAL, "%s: b must lie in [0, tokens]", fn);
    if (!d_k || !d_v || !w_k || !w_v) return fail(KVFIX_EINVAL, "%s: d_k, d_v, w_k, w_v are required", fn);
    if (b > 0 && (!idx_k || !idx_v)) return fail(KVFIX_EINVAL, "%s: idx_k and idx_v are required when b > 0", fn);
    if (units > 0 && !delta) return fail(KVFIX_EINVAL, "%s: delta is null", fn);
    if (!(rope_base > 1.0) || !isfinite(rope_base)) return fail(KVFIX_EINVAL, "%s: rope_base must be finite and > 1", fn);
    cudaStream_t s = (cudaStream_t)stream;
    RopeTheta th = make_theta(rope_base, reuse.head_dim);
    cudaError_t e = launch_score(k_reuse, v_reuse, reuse, k_fresh, v_fresh, fresh, agents, delta, th,
                                 d_k, d_v, w_k, w_v, mask_union, s);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    e = launch_select_f32(d_k, d_v, (int)units, n, b, idx_k, idx_v, mask_k, mask_v, mask_union, s);
    return launched(e, fn);
}

kvfix_status kvfix_mean_correct(const kvfix_bf16* k_reuse, const kvfix_bf16* v_reuse,
                                kvfix_kv_desc reuse, const kvfix_bf16* k_fresh,
                                const kvfix_bf16* v_fresh, kvfix_kv_desc fresh, kvfix_bf16* k_out,
                                kvfix_bf16* v_out, kvfix_kv_desc out, int32_t agents,
                                const int32_t* delta, double rope_base, const int32_t* idx_k,
                                const int32_t* idx_v, int32_t b, const float* w_k,
                                const float* w_v, float* mu_k, float* mu_v, void* stream) {
    const char* fn = "kvfix_mean_correct";
    if (agents < 1) return fail(KVFIX_EINVAL, "%s: agents must be >= 1", fn);
    if (!same_shape(reuse, fresh) || !same_shape(reuse, out))
        return fail(KVFIX_EINVAL, "%s: reuse, fresh and out shapes differ", fn);
    const long long units = (long long)agents * reuse.chunks;
    if (fresh.chunks != units || out.chunks != units)
        return fail(KVFIX_EINVAL, "%s: fresh.chunks and out.chunks must equal agents*reuse.chunks", fn);
    if (units > 65535 || reuse.layers > 65535 || reuse.chunks > 65535)
        return fail(KVFIX_EINVAL, "%s: at most 65535 units and 65535 layers", fn);
    if ((long long)reuse.kv_heads * reuse.head_dim > 4096)
        return fail(KVFIX_EINVAL, "%s: kv_heads*head_dim must be <= 4096", fn);
    if (b < 0 || b > reuse.tokens) return fail(KVFIX_EINVAL, "%s: b must lie in [0, tokens]", fn);
    if (!(rope_base > 1.0) || !isfinite(rope_base)) return fail(KVFIX_EINVAL, "%s: rope_base must be finite and > 1", fn);
    if (units > 0 && !delta) return fail(KVFIX_EINVAL, "%s: delta is null", fn);
    struct PlaneArgs {
        const kvfix_bf16* reuse;
        const kvfix_bf16* fresh;
        kvfix_bf16* out;
        const int32_t* idx;
        const float* w;
        float* mu;
        bool rotate;
        const char* name;
    } planes[2] = {{k_reuse, k_fresh, k_out, idx_k, w_k, mu_k, true, "K"},
                   {v_reuse, v_fresh, v_out, idx_v, w_v, mu_v, false, "V"}};
    kvfix_status st;
    int active = 0;
    for (auto& p : planes) {
        if (!p.reuse && !p.fresh && !p.out) continue;
        ++active;
        char what[96];
        snprintf(what, sizeof what, "%s: %s reuse", fn, p.name);
        if ((st = check_plane(p.reuse, reuse, what)) != KVFIX_OK) return st;
        snprintf(what, sizeof what, "%s: %s fresh", fn, p.name);
        if ((st = check_plane(p.fresh, fresh, what)) != KVFIX_OK) return st;
        snprintf(what, sizeof what, "%s: %s out", fn, p.name);
        if ((st = check_plane(p.out, out, what)) != KVFIX_OK) return st;
        if (!p.w || !p.mu || (b > 0 && !p.idx))
            return fail(KVFIX_EINVAL, "%s: %s plane needs w, mu and (b > 0) idx", fn, p.name);
        if (overlaps(p.out, out, p.reuse, reuse) || overlaps(p.out, out, p.fresh, fresh))
            return fail(KVFIX_EINVAL, "%s: %s out overlaps an input", fn, p.name);
        const size_t mu_bytes = sizeof(float) * (size_t)units * reuse.layers * reuse.kv_heads * reuse.head_dim;
        if (overlaps_bytes(p.mu, mu_bytes, p.w, sizeof(float) * (size_t)units * reuse.tokens))
            return fail(KVFIX_EINVAL, "%s: %s mu overlaps w", fn, p.name);
        uintptr_t o0, o1;
        extent(p.out, out, &o0, &o1);
        if (overlaps_bytes(p.mu, mu_bytes, (const void*)o0, o1 - o0))
            return fail(KVFIX_EINVAL, "%s: %s mu overlaps out", fn, p.name);
    }
    if (!active) return fail(KVFIX_EINVAL, "%s: no plane given", fn);
    cudaStream_t s = (cudaStream_t)stream;
    RopeTheta th = make_theta(rope_base, reuse.head_dim);
    McPlanes mp;
    for (int q = 0; q < 2; ++q) {
        mp.reuse[q] = planes[q].reuse;
        mp.fresh[q] = planes[q].fresh;
        mp.out[q] = planes[q].out;
        mp.idx[q] = planes[q].idx;
        mp.w[q] = planes[q].w;
        mp.mu[q] = planes[q].mu;
    }
    return launched(launch_mean_correct(mp, reuse, fresh, out, agents, delta, th, b, s), fn);
}

kvfix_status kvfix_lowrank_apply(const kvfix_bf16* x, kvfix_kv_desc desc, const kvfix_bf16* A,
                                 const kvfix_bf16* B, int32_t rank, kvfix_bf16* out,
                                 kvfix_kv_desc out_desc, void* stream) {
    const char* fn = "kvfix_lowrank_apply";
    kvfix_status st;
    if ((st = check_plane(x, desc, "kvfix_lowrank_apply: x")) != KVFIX_OK) return st;
    if ((st = check_plane(out, out_desc, "kvfix_lowrank_apply: out")) != KVFIX_OK) return st;
    if (!same_shape(desc, out_desc) || desc.chunks != out_desc.chunks)
        return fail(KVFIX_EINVAL, "%s: x and out shapes differ", fn);
    if (!A || !B) return fail(KVFIX_EINVAL, "%s: A and B are required", fn);
    if (!aligned16(A) || !aligned16(B)) return fail(KVFIX_EINVAL, "%s: A and B must be 16-byte aligned", fn);
    if (rank != 16 && rank != 32 && rank != 64) return fail(KVFIX_EINVAL, "%s: rank must be 16, 32 or 64", fn);
    if (desc.tokens > 0 && ((long long)desc.chunks * desc.layers * desc.kv_heads * desc.tokens >= (1ll << 31)))
        return fail(KVFIX_EINVAL, "%s: at most 2^31 factor rows", fn);
    if (desc.head_dim != 64 && desc.head_dim != 128) return fail(KVFIX_EINVAL, "%s: head_dim must be 64 or 128", fn);
    const bool in_place = (const void*)x == (const void*)out && same_desc(desc, out_desc);
    if (!in_place && overlaps(x, desc, out, out_desc))
        return fail(KVFIX_EINVAL, "%s: out overlaps x (only an exact in-place call is allowed)", fn);
    const size_t na = 2 * (size_t)desc.chunks * desc.layers * desc.kv_heads * desc.tokens * rank;
    const size_t nb = 2 * (size_t)desc.chunks * desc.layers * desc.kv_heads * rank * desc.head_dim;
    uintptr_t o0, o1;
    extent(out, out_desc, &o0, &o1);
    if (overlaps_bytes((const void*)o0, o1 - o0, A, na) || overlaps_bytes((const void*)o0, o1 - o0, B, nb))
        return fail(KVFIX_EINVAL, "%s: out overlaps A or B", fn);
    return launched(launch_lowrank(x, desc, A, B, rank, out, out_desc, (cudaStream_t)stream), fn);
}

size_t kvfix_draft_rank_workspace_bytes(kvfix_kv_desc desc, int32_t layer_begin) {
    return draft_workspace_bytes(desc, layer_begin);
}

kvfix_status kvfix_draft_rank(const kvfix_bf16* k, kvfix_kv_desc desc, const kvfix_bf16* q,
                              int32_t draft_steps, int32_t q_heads, int32_t layer_begin,
                              int32_t k_rows, int32_t* idx, double* scores,
                              const kvfix_bf16* k_fresh, const kvfix_bf16* v_fresh,
                              kvfix_kv_desc fresh_desc, kvfix_bf16* k_io, kvfix_bf16* v_io,
                              void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "kvfix_draft_rank";
    kvfix_status st;
    if ((st = check_plane(k, desc, "kvfix_draft_rank: k")) != KVFIX_OK) return st;
    if (!q || !aligned16(q)) return fail(KVFIX_EINVAL, "%s: q must be a 16-byte aligned device pointer", fn);
    if (desc.head_dim != 64 && desc.head_dim != 128) return fail(KVFIX_EINVAL, "%s: head_dim must be 64 or 128", fn);
    if (draft_steps < 1 || q_heads < 1 || q_heads % desc.kv_heads)
        return fail(KVFIX_EINVAL, "%s: q_heads must be a positive multiple of kv_heads, draft_steps >= 1", fn);
    if ((q_heads / desc.kv_heads) * draft_steps > 16)
        return fail(KVFIX_EINVAL, "%s: (q_heads/kv_heads)*draft_steps must be <= 16", fn);
    if (layer_begin < 0 || layer_begin > desc.layers) return fail(KVFIX_EINVAL, "%s: layer_begin out of range", fn);
    if (desc.tokens > 16384 || desc.chunks > 65535) return fail(KVFIX_EINVAL, "%s: tokens <= 16384, chunks <= 65535", fn);
    if ((long long)desc.chunks * (desc.layers - layer_begin) * desc.kv_heads > 65535)
        return fail(KVFIX_EINVAL, "%s: at most 65535 (chunk, layer, head) units", fn);
    if (k_rows < 0 || k_rows > desc.tokens) return fail(KVFIX_EINVAL, "%s: k_rows must lie in [0, tokens]", fn);
    if (!scores || (k_rows > 0 && !idx)) return fail(KVFIX_EINVAL, "%s: scores and idx are required", fn);
    if (workspace_bytes < draft_workspace_bytes(desc, layer_begin) || (!workspace && workspace_bytes))
        return fail(KVFIX_EINVAL, "%s: workspace smaller than kvfix_draft_rank_workspace_bytes()", fn);
    if (workspace && !aligned16(workspace)) return fail(KVFIX_EINVAL, "%s: workspace not 16-byte aligned", fn);
    if (k_io || v_io) {
        if ((k_io && !k_fresh) || (v_io && !v_fresh)) return fail(KVFIX_EINVAL, "%s: k_io/v_io need k_fresh/v_fresh", fn);
        if (k_io && (st = check_plane(k_io, desc, "kvfix_draft_rank: k_io")) != KVFIX_OK) return st;
        if (v_io && (st = check_plane(v_io, desc, "kvfix_draft_rank: v_io")) != KVFIX_OK) return st;
        if (k_fresh && (st = check_plane(k_fresh, fresh_desc, "kvfix_draft_rank: k_fresh")) != KVFIX_OK) return st;
        if (v_fresh && (st = check_plane(v_fresh, fresh_desc, "kvfix_draft_rank: v_fresh")) != KVFIX_OK) return st;
        if (!same_shape(desc, fresh_desc) || fresh_desc.chunks != desc.chunks)
            return fail(KVFIX_EINVAL, "%s: fresh_desc must match desc", fn);
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_draft(k, desc, q, draft_steps, q_heads, layer_begin, k_rows, idx, scores, workspace, s);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (k_io) {
        if ((e = launch_row_repair(k_io, desc, k_fresh, fresh_desc, idx, k_rows, s)) != cudaSuccess) return cuda_fail(e, fn);
    }
    if (v_io) {
        if ((e = launch_row_repair(v_io, desc, v_fresh, fresh_desc, idx, k_rows, s)) != cudaSuccess) return cuda_fail(e, fn);
    }
    return KVFIX_OK;
}

size_t kvfix_lowrank_draft_workspace_bytes(kvfix_kv_desc desc, int32_t layer_begin) {
    return lowrank_draft_workspace_bytes(desc, layer_begin);
}

kvfix_status kvfix_lowrank_draft(const kvfix_bf16* x, kvfix_kv_desc desc, const kvfix_bf16* A, const kvfix_bf16* B,
                                 int32_t rank, kvfix_bf16* out, kvfix_kv_desc out_desc, const kvfix_bf16* q,
                                 int32_t draft_steps, int32_t q_heads, int32_t layer_begin, int32_t k_rows,
                                 int32_t* idx, double* scores, const kvfix_bf16* k_fresh, const kvfix_bf16* v_fresh,
                                 kvfix_kv_desc fresh_desc, kvfix_bf16* v_io, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    const char* fn = "kvfix_lowrank_draft";
    kvfix_status st;
    // the low-rank part: the checks of kvfix_lowrank_apply
    if ((st = check_plane(x, desc, "kvfix_lowrank_draft: x")) != KVFIX_OK) return st;
    if ((st = check_plane(out, out_desc, "kvfix_lowrank_draft: out")) != KVFIX_OK) return st;
    if (!same_shape(desc, out_desc) || desc.chunks != out_desc.chunks)
        return fail(KVFIX_EINVAL, "%s: x and out shapes differ", fn);
    if (!A || !B) return fail(KVFIX_EINVAL, "%s: A and B are required", fn);
    if (!aligned16(A) || !aligned16(B)) return fail(KVFIX_EINVAL, "%s: A and B must be 16-byte aligned", fn);
    if (rank != 16 && rank != 32 && rank != 64) return fail(KVFIX_EINVAL, "%s: rank must be 16, 32 or 64", fn);
    if (desc.tokens > 0 && ((long long)desc.chunks * desc.layers * desc.kv_heads * desc.tokens >= (1ll << 31)))
        return fail(KVFIX_EINVAL, "%s: at most 2^31 factor rows", fn);
    if (desc.head_dim != 64 && desc.head_dim != 128) return fail(KVFIX_EINVAL, "%s: head_dim must be 64 or 128", fn);
    const bool in_place = (const void*)x == (const void*)out && same_desc(desc, out_desc);
    if (!in_place && overlaps(x, desc, out, out_desc))
        return fail(KVFIX_EINVAL, "%s: out overlaps x (only an exact in-place call is allowed)", fn);
    const size_t na = 2 * (size_t)desc.chunks * desc.layers * desc.kv_heads * desc.tokens * rank;
    const size_t nb = 2 * (size_t)desc.chunks * desc.layers * desc.kv_heads * rank * desc.head_dim;
    uintptr_t o0, o1;
    extent(out, out_desc, &o0, &o1);
    if (overlaps_bytes((const void*)o0, o1 - o0, A, na) || overlaps_bytes((const void*)o0, o1 - o0, B, nb))
        return fail(KVFIX_EINVAL, "%s: out overlaps A or B", fn);
    // the draft part: the checks of kvfix_draft_rank, on the corrected plane
    if (!q || !aligned16(q)) return fail(KVFIX_EINVAL, "%s: q must be a 16-byte aligned device pointer", fn);
    if (draft_steps < 1 || q_heads < 1 || q_heads % desc.kv_heads)
        return fail(KVFIX_EINVAL, "%s: q_heads must be a positive multiple of kv_heads, draft_steps >= 1", fn);
    if ((q_heads / desc.kv_heads) * draft_steps > 16)
        return fail(KVFIX_EINVAL, "%s: (q_heads/kv_heads)*draft_steps must be <= 16", fn);
    if (layer_begin < 0 || layer_begin > desc.layers) return fail(KVFIX_EINVAL, "%s: layer_begin out of range", fn);
    if (desc.tokens > 16384 || desc.chunks > 65535) return fail(KVFIX_EINVAL, "%s: tokens <= 16384, chunks <= 65535", fn);
    if (k_rows < 0 || k_rows > desc.tokens) return fail(KVFIX_EINVAL, "%s: k_rows must lie in [0, tokens]", fn);
    if (!scores || (k_rows > 0 && !idx)) return fail(KVFIX_EINVAL, "%s: scores and idx are required", fn);
    if (!workspace || workspace_bytes < lowrank_draft_workspace_bytes(desc, layer_begin))
        return fail(KVFIX_EINVAL, "%s: workspace smaller than kvfix_lowrank_draft_workspace_bytes()", fn);
    if (!aligned16(workspace)) return fail(KVFIX_EINVAL, "%s: workspace not 16-byte aligned", fn);
    if (k_fresh || v_io || v_fresh) {
        if (v_io && !v_fresh) return fail(KVFIX_EINVAL, "%s: v_io needs v_fresh", fn);
        if (k_fresh && (st = check_plane(k_fresh, fresh_desc, "kvfix_lowrank_draft: k_fresh")) != KVFIX_OK) return st;
        if (v_fresh && (st = check_plane(v_fresh, fresh_desc, "kvfix_lowrank_draft: v_fresh")) != KVFIX_OK) return st;
        if (v_io && (st = check_plane(v_io, out_desc, "kvfix_lowrank_draft: v_io")) != KVFIX_OK) return st;
        if (!same_shape(desc, fresh_desc) || fresh_desc.chunks != desc.chunks)
            return fail(KVFIX_EINVAL, "%s: fresh_desc must match desc", fn);
        if (k_fresh && overlaps(out, out_desc, k_fresh, fresh_desc)) return fail(KVFIX_EINVAL, "%s: out overlaps k_fresh", fn);
        if (v_io && overlaps(out, out_desc, v_io, out_desc)) return fail(KVFIX_EINVAL, "%s: v_io overlaps out", fn);
    }
    if (workspace && overlaps_bytes(workspace, workspace_bytes, (const void*)o0, o1 - o0))
        return fail(KVFIX_EINVAL, "%s: workspace overlaps out", fn);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_lowrank_draft(x, desc, A, B, rank, out, out_desc, q, draft_steps, q_heads, layer_begin,
                                         k_rows, idx, scores, workspace, s);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (k_fresh && (e = launch_row_repair(out, out_desc, k_fresh, fresh_desc, idx, k_rows, s)) != cudaSuccess)
        return cuda_fail(e, fn);
    if (v_io && (e = launch_row_repair(v_io, out_desc, v_fresh, fresh_desc, idx, k_rows, s)) != cudaSuccess)
        return cuda_fail(e, fn);
    return KVFIX_OK;
}

kvfix_status kvfix_diff_encode(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                               kvfix_kv_desc master, const kvfix_bf16* sib_k,
                               const kvfix_bf16* sib_v, kvfix_kv_desc sib, int32_t block_tokens,
                               uint32_t* mask, int64_t* offsets, kvfix_bf16* payload,
                               int64_t capacity_entries, int64_t* h_entries, void* stream) {
    const char* fn = "kvfix_diff_encode";
    kvfix_status st;
    if ((st = check_plane(master_k, master, "kvfix_diff_encode: master_k")) != KVFIX_OK) return st;
    if ((st = check_plane(master_v, master, "kvfix_diff_encode: master_v")) != KVFIX_OK) return st;
    if ((st = check_plane(sib_k, sib, "kvfix_diff_encode: sib_k")) != KVFIX_OK) return st;
    if ((st = check_plane(sib_v, sib, "kvfix_diff_encode: sib_v")) != KVFIX_OK) return st;
    if (master.chunks != 1) return fail(KVFIX_EINVAL, "%s: master.chunks must be 1", fn);
    if (!same_shape(master, sib)) return fail(KVFIX_EINVAL, "%s: master and sibling shapes differ", fn);
    if (block_tokens < 1 || master.tokens % block_tokens)
        return fail(KVFIX_EINVAL, "%s: block_tokens must divide tokens", fn);
    if (!mask || !offsets) return fail(KVFIX_EINVAL, "%s: mask and offsets are required", fn);
    if (capacity_entries < 0) return fail(KVFIX_EINVAL, "%s: negative capacity", fn);
    if (capacity_entries > 0 && (!payload || !aligned16(payload)))
        return fail(KVFIX_EINVAL, "%s: payload must be a 16-byte aligned device pointer", fn);
    const long long per_sibling = (long long)master.layers * (master.tokens / block_tokens);
    const long long entries = per_sibling * sib.chunks;
    if (entries >= (1ll << 31)) return fail(KVFIX_EINVAL, "%s: too many entries", fn);
    if (sib.chunks > 65535 || master.layers > 65535) return fail(KVFIX_EINVAL, "%s: at most 65535 siblings and layers", fn);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(mask, 0, sizeof(uint32_t) * (size_t)((entries + 31) / 32), s);
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if ((e = launch_diff_mask(master_k, master_v, master, sib_k, sib_v, sib, block_tokens, mask, s)) != cudaSuccess)
        return cuda_fail(e, fn);
    if ((e = launch_diff_scan(mask, sib.chunks, per_sibling, offsets, s)) != cudaSuccess) return cuda_fail(e, fn);
    if (h_entries) {
        int64_t total = 0;
        if ((e = cudaMemcpyAsync(&total, offsets + entries, sizeof total, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e, fn);
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, fn);
        *h_entries = total;
        if (total > capacity_entries)
            return fail(KVFIX_ENOSPACE, "%s: %lld entries needed, capacity %lld", fn, (long long)total,
                        (long long)capacity_entries);
    }
    if (capacity_entries == 0) return KVFIX_OK;
    return launched(launch_diff_pack(sib_k, sib_v, sib, block_tokens, mask, offsets, payload,
                                     capacity_entries, s), fn);
}

kvfix_status kvfix_diff_gather(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                               kvfix_kv_desc master, const uint32_t* mask,
                               const int64_t* offsets, const kvfix_bf16* payload,
                               int64_t payload_entries, int32_t siblings, int32_t block_tokens,
                               kvfix_bf16* out_k, kvfix_bf16* out_v, kvfix_kv_desc out,
                               void* stream) {
    const char* fn = "kvfix_diff_gather";
    kvfix_status st;
    if ((st = check_plane(master_k, master, "kvfix_diff_gather: master_k")) != KVFIX_OK) return st;
    if ((st = check_plane(master_v, master, "kvfix_diff_gather: master_v")) != KVFIX_OK) return st;
    if ((st = check_plane(out_k, out, "kvfix_diff_gather: out_k")) != KVFIX_OK) return st;
    if ((st = check_plane(out_v, out, "kvfix_diff_gather: out_v")) != KVFIX_OK) return st;
    if (master.chunks != 1) return fail(KVFIX_EINVAL, "%s: master.chunks must be 1", fn);
    if (!same_shape(master, out) || out.chunks != siblings)
        return fail(KVFIX_EINVAL, "%s: out must have `siblings` chunks of the master's shape", fn);
    if (block_tokens < 1 || master.tokens % block_tokens)
        return fail(KVFIX_EINVAL, "%s: block_tokens must divide tokens", fn);
    if (siblings < 0 || siblings > 65535 || master.layers > 65535)
        return fail(KVFIX_EINVAL, "%s: siblings and layers must be <= 65535", fn);
    if (!mask || !offsets) return fail(KVFIX_EINVAL, "%s: mask and offsets are required", fn);
    if (payload_entries < 0) return fail(KVFIX_EINVAL, "%s: negative payload_entries", fn);
    if (payload_entries > 0 && (!payload || !aligned16(payload)))
        return fail(KVFIX_EINVAL, "%s: payload must be a 16-byte aligned device pointer", fn);
    if (overlaps(out_k, out, master_k, master) || overlaps(out_v, out, master_v, master) ||
        overlaps(out_k, out, out_v, out))
        return fail(KVFIX_EINVAL, "%s: outputs overlap the master or each other", fn);
    return launched(launch_diff_gather(master_k, master_v, master, mask, offsets, payload,
                                       payload_entries, siblings, block_tokens, out_k, out_v, out,
                                       (cudaStream_t)stream), fn);
}

// Shared by the joint and the per-plane restore: with mask_v set, (mask, offsets, payload,
// payload_entries) is the key plane's list and (mask_v, offsets_v, payload_v, entries_v) the
// value plane's; otherwise one list holds both planes.
static kvfix_status restore_impl(const char* fn, const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                                 kvfix_kv_desc master, const uint32_t* mask, const int64_t* offsets,
                                 const kvfix_bf16* payload, int64_t payload_entries, const uint32_t* mask_v,
                                 const int64_t* offsets_v, const kvfix_bf16* payload_v, int64_t entries_v,
                                 bool split, int32_t siblings, int32_t block_tokens, const int32_t* delta,
                                 double rope_base, const int32_t* slot_mapping, kvfix_bf16* pool_k,
                                 kvfix_bf16* pool_v, kvfix_kv_desc pool, void* stream) {
    kvfix_status st;
    char what[64];
    const void* planes[4] = {master_k, master_v, pool_k, pool_v};
    const char* names[4] = {"master_k", "master_v", "pool_k", "pool_v"};
    for (int i = 0; i < 4; ++i) {
        snprintf(what, sizeof what, "%s: %s", fn, names[i]);
        if ((st = check_plane(planes[i], i < 2 ? master : pool, what)) != KVFIX_OK) return st;
    }
    if (master.chunks != 1 || pool.chunks != 1)
        return fail(KVFIX_EINVAL, "%s: master.chunks and pool.chunks must be 1", fn);
    if (pool.layers != master.layers || pool.kv_heads != master.kv_heads ||
        pool.head_dim != master.head_dim)
        return fail(KVFIX_EINVAL, "%s: the pool must have the master's layers, heads and head_dim", fn);
    if (block_tokens < 1 || master.tokens % block_tokens)
        return fail(KVFIX_EINVAL, "%s: block_tokens must divide tokens", fn);
    if (siblings < 0 || siblings > 65535 || master.layers > 65535)
        return fail(KVFIX_EINVAL, "%s: siblings and layers must be <= 65535", fn);
    if (!mask || !offsets || (split && (!mask_v || !offsets_v)))
        return fail(KVFIX_EINVAL, "%s: every mask and offset array is required", fn);
    if (siblings > 0 && (!delta || (master.tokens > 0 && !slot_mapping)))
        return fail(KVFIX_EINVAL, "%s: delta and slot_mapping are required", fn);
    if (!(rope_base > 1.0) || !isfinite(rope_base))
        return fail(KVFIX_EINVAL, "%s: rope_base must be finite and > 1", fn);
    if (payload_entries < 0 || entries_v < 0) return fail(KVFIX_EINVAL, "%s: negative payload entries", fn);
    if ((payload_entries > 0 && (!payload || !aligned16(payload))) ||
        (split && entries_v > 0 && (!payload_v || !aligned16(payload_v))))
        return fail(KVFIX_EINVAL, "%s: payloads must be 16-byte aligned device pointers", fn);
    if (overlaps(pool_k, pool, master_k, master) || overlaps(pool_v, pool, master_v, master) ||
        overlaps(pool_k, pool, master_v, master) || overlaps(pool_v, pool, master_k, master) ||
        overlaps(pool_k, pool, pool_v, pool))
        return fail(KVFIX_EINVAL, "%s: pool planes overlap the master or each other", fn);
    RopeTheta th = make_theta(rope_base, master.head_dim);
    return launched(launch_diff_restore(master_k, master_v, master, mask, offsets, payload, payload_entries,
                                        siblings, block_tokens, delta, th, slot_mapping, pool_k, pool_v, pool,
                                        (cudaStream_t)stream, split ? mask_v : nullptr, offsets_v, payload_v,
                                        split ? entries_v : 0),
                    fn);
}

kvfix_status kvfix_diff_restore(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                                kvfix_kv_desc master, const uint32_t* mask,
                                const int64_t* offsets, const kvfix_bf16* payload,
                                int64_t payload_entries, int32_t siblings, int32_t block_tokens,
                                const int32_t* delta, double rope_base,
                                const int32_t* slot_mapping, kvfix_bf16* pool_k,
                                kvfix_bf16* pool_v, kvfix_kv_desc pool, void* stream) {
    return restore_impl("kvfix_diff_restore", master_k, master_v, master, mask, offsets, payload, payload_entries,
                        nullptr, nullptr, nullptr, 0, false, siblings, block_tokens, delta, rope_base,
                        slot_mapping, pool_k, pool_v, pool, stream);
}

kvfix_status kvfix_diff_restore_split(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                                      kvfix_kv_desc master, const uint32_t* mask_k, const uint32_t* mask_v,
                                      const int64_t* offsets_k, const int64_t* offsets_v,
                                      const kvfix_bf16* payload_k, const kvfix_bf16* payload_v, int64_t entries_k,
                                      int64_t entries_v, int32_t siblings, int32_t block_tokens,
                                      const int32_t* delta, double rope_base, const int32_t* slot_mapping,
                                      kvfix_bf16* pool_k, kvfix_bf16* pool_v, kvfix_kv_desc pool, void* stream) {
    return restore_impl("kvfix_diff_restore_split", master_k, master_v, master, mask_k, offsets_k, payload_k,
                        entries_k, mask_v, offsets_v, payload_v, entries_v, true, siblings, block_tokens, delta,
                        rope_base, slot_mapping, pool_k, pool_v, pool, stream);
}

static kvfix_status check_factor(const void* p, const char* fn, const char* name) {
    if (!p) return fail(KVFIX_EINVAL, "%s: %s is null", fn, name);
    if (!aligned16(p)) return fail(KVFIX_EINVAL, "%s: %s not 16-byte aligned", fn, name);
    return KVFIX_OK;
}

static kvfix_status check_anchor_shape(const kvfix_kv_desc& d, int32_t anchors, int32_t rank, int head_dim,
                                       const char* fn) {
    if (anchors < 1 || anchors > 16) return fail(KVFIX_EINVAL, "%s: anchors must be in [1, 16]", fn);
    if (rank != 16 && rank != 32 && rank != 64) return fail(KVFIX_EINVAL, "%s: rank must be 16, 32 or 64", fn);
    if ((d.kv_heads * d.head_dim) % 128 != 0)
        return fail(KVFIX_EINVAL, "%s: kv_heads * head_dim must be a multiple of 128", fn);
    if (!anchor_shape_ok(anchors, rank, head_dim))
        return fail(KVFIX_EINVAL, "%s: %d anchors of rank %d do not fit in shared memory", fn, anchors, rank);
    const long long rows = (long long)d.chunks * anchors * d.layers *
                           (long long)(d.tokens > d.kv_heads * d.head_dim ? d.tokens : d.kv_heads * d.head_dim);
    if (rows >= (1ll << 31)) return fail(KVFIX_EINVAL, "%s: factor rows exceed 2^31", fn);
    if (d.layers > 65535 || d.chunks > 32767) return fail(KVFIX_EINVAL, "%s: too many layers or segments", fn);
    return KVFIX_OK;
}

size_t kvfix_anchor_gate_workspace_bytes(kvfix_kv_desc src, int32_t anchors, int32_t prefix) {
    if (anchors < 1 || prefix < 1 || src.chunks < 0 || src.layers < 0) return 0;
    return anchor_gate_workspace_bytes(src, anchors, prefix);
}

kvfix_status kvfix_anchor_gate(const kvfix_bf16* v_src, kvfix_kv_desc src, const kvfix_bf16* a_c,
                               const kvfix_bf16* b_ct, int32_t anchors, int32_t rank, int32_t prefix,
                               double temperature, double tau, double* d, double* g, double* hbar,
                               int32_t* accept, void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "kvfix_anchor_gate";
    kvfix_status st;
    if ((st = check_plane(v_src, src, "kvfix_anchor_gate: v_src")) != KVFIX_OK) return st;
    if ((st = check_anchor_shape(src, anchors, rank, 0, fn)) != KVFIX_OK) return st;
    if (prefix < 1 || prefix > src.tokens) return fail(KVFIX_EINVAL, "%s: prefix must be in [1, tokens]", fn);
    if (!(temperature > 0.0) || !isfinite(temperature) || isnan(tau))
        return fail(KVFIX_EINVAL, "%s: temperature must be finite and > 0, tau a number", fn);
    if ((st = check_factor(a_c, fn, "a_c")) != KVFIX_OK) return st;
    if ((st = check_factor(b_ct, fn, "b_ct")) != KVFIX_OK) return st;
    if (!d || !g || !hbar || !accept) return fail(KVFIX_EINVAL, "%s: d, g, hbar and accept are required", fn);
    if (src.chunks > 0 && src.layers > 0) {
        if (!workspace || workspace_bytes < anchor_gate_workspace_bytes(src, anchors, prefix))
            return fail(KVFIX_EINVAL, "%s: workspace smaller than kvfix_anchor_gate_workspace_bytes()", fn);
        if (!aligned16(workspace)) return fail(KVFIX_EINVAL, "%s: workspace not 16-byte aligned", fn);
    }
    if (src.layers == 0) return fail(KVFIX_EINVAL, "%s: no layers", fn);
    return launched(launch_anchor_gate(v_src, src, a_c, b_ct, anchors, rank, prefix, temperature, tau, d, g, hbar,
                                       accept, workspace, (cudaStream_t)stream),
                    fn);
}

static kvfix_status anchor_correct_impl(const char* fn, const kvfix_bf16* k_src, const kvfix_bf16* v_src,
                                        kvfix_kv_desc src, const kvfix_bf16* a_c_k, const kvfix_bf16* b_ct_k,
                                        const kvfix_bf16* a_c_v, const kvfix_bf16* b_ct_v, const kvfix_bf16* a_d_k,
                                        const kvfix_bf16* b_dt_k, const kvfix_bf16* a_d_v, const kvfix_bf16* b_dt_v,
                                        int32_t anchors, int32_t rank, double temperature, const int32_t* delta,
                                        double rope_base, const int32_t* accept, float* w_k, float* w_v,
                                        kvfix_bf16* k_out, kvfix_bf16* v_out, kvfix_kv_desc out, void* stream,
                                        const AnchorGateOut* gate) {
    kvfix_status st;
    if ((st = check_plane(k_src, src, "anchor correction: k_src")) != KVFIX_OK) return st;
    if ((st = check_plane(v_src, src, "anchor correction: v_src")) != KVFIX_OK) return st;
    if ((st = check_plane(k_out, out, "anchor correction: k_out")) != KVFIX_OK) return st;
    if ((st = check_plane(v_out, out, "anchor correction: v_out")) != KVFIX_OK) return st;
    if (!same_shape(src, out) || src.chunks != out.chunks)
        return fail(KVFIX_EINVAL, "%s: out must have the shape of src", fn);
    if (src.head_dim != 64 && src.head_dim != 128) return fail(KVFIX_EINVAL, "%s: head_dim must be 64 or 128", fn);
    if ((st = check_anchor_shape(src, anchors, rank, src.head_dim, fn)) != KVFIX_OK) return st;
    if (!(temperature > 0.0) || !isfinite(temperature))
        return fail(KVFIX_EINVAL, "%s: temperature must be finite and > 0", fn);
    if (!(rope_base > 1.0) || !isfinite(rope_base))
        return fail(KVFIX_EINVAL, "%s: rope_base must be finite and > 1", fn);
    const void* f[8] = {a_c_k, b_ct_k, a_c_v, b_ct_v, a_d_k, b_dt_k, a_d_v, b_dt_v};
    const char* names[8] = {"a_c_k", "b_ct_k", "a_c_v", "b_ct_v", "a_d_k", "b_dt_k", "a_d_v", "b_dt_v"};
    for (int i = 0; i < 8; ++i)
        if ((st = check_factor(f[i], fn, names[i])) != KVFIX_OK) return st;
    if (src.chunks > 0 && (!delta || !w_k || !w_v))
        return fail(KVFIX_EINVAL, "%s: delta, w_k and w_v are required", fn);
    const bool k_in_place = (const void*)k_src == (const void*)k_out && same_desc(src, out);
    const bool v_in_place = (const void*)v_src == (const void*)v_out && same_desc(src, out);
    if ((!k_in_place && overlaps(k_out, out, k_src, src)) || (!v_in_place && overlaps(v_out, out, v_src, src)) ||
        overlaps(k_out, out, v_src, src) || overlaps(v_out, out, k_src, src) || overlaps(k_out, out, v_out, out))
        return fail(KVFIX_EINVAL, "%s: outputs overlap the sources (other than exactly in place) or each other", fn);
    AnchorPlanes pl;
    pl.src[0] = k_src;
    pl.src[1] = v_src;
    pl.ac[0] = a_c_k;
    pl.ac[1] = a_c_v;
    pl.bct[0] = b_ct_k;
    pl.bct[1] = b_ct_v;
    pl.ad[0] = a_d_k;
    pl.ad[1] = a_d_v;
    pl.bdt[0] = b_dt_k;
    pl.bdt[1] = b_dt_v;
    pl.w[0] = w_k;
    pl.w[1] = w_v;
    pl.out[0] = k_out;
    pl.out[1] = v_out;
    RopeTheta th = make_theta(rope_base, src.head_dim);
    return launched(launch_anchor_correct(pl, src, out, anchors, rank, temperature, delta, th, accept,
                                          (cudaStream_t)stream, gate),
                    fn);
}

kvfix_status kvfix_anchor_correct(const kvfix_bf16* k_src, const kvfix_bf16* v_src, kvfix_kv_desc src,
                                  const kvfix_bf16* a_c_k, const kvfix_bf16* b_ct_k, const kvfix_bf16* a_c_v,
                                  const kvfix_bf16* b_ct_v, const kvfix_bf16* a_d_k, const kvfix_bf16* b_dt_k,
                                  const kvfix_bf16* a_d_v, const kvfix_bf16* b_dt_v, int32_t anchors,
                                  int32_t rank, double temperature, const int32_t* delta, double rope_base,
                                  const int32_t* accept, float* w_k, float* w_v, kvfix_bf16* k_out,
                                  kvfix_bf16* v_out, kvfix_kv_desc out, void* stream) {
    return anchor_correct_impl("kvfix_anchor_correct", k_src, v_src, src, a_c_k, b_ct_k, a_c_v, b_ct_v, a_d_k, b_dt_k,
                               a_d_v, b_dt_v, anchors, rank, temperature, delta, rope_base, accept, w_k, w_v, k_out,
                               v_out, out, stream, nullptr);
}

kvfix_status kvfix_anchor_gate_correct(const kvfix_bf16* k_src, const kvfix_bf16* v_src, kvfix_kv_desc src,
                                       const kvfix_bf16* a_c_k, const kvfix_bf16* b_ct_k, const kvfix_bf16* a_c_v,
                                       const kvfix_bf16* b_ct_v, const kvfix_bf16* a_d_k, const kvfix_bf16* b_dt_k,
                                       const kvfix_bf16* a_d_v, const kvfix_bf16* b_dt_v, int32_t anchors,
                                       int32_t rank, int32_t prefix, double temperature, double tau,
                                       const int32_t* delta, double rope_base, double* d, double* g, double* hbar,
                                       int32_t* accept, float* w_k, float* w_v, kvfix_bf16* k_out, kvfix_bf16* v_out,
                                       kvfix_kv_desc out, void* workspace, size_t workspace_bytes, void* stream) {
    const char* fn = "kvfix_anchor_gate_correct";
    if (prefix < 1 || prefix > src.tokens) return fail(KVFIX_EINVAL, "%s: prefix must be in [1, tokens]", fn);
    if (isnan(tau)) return fail(KVFIX_EINVAL, "%s: tau must be a number", fn);
    if (src.chunks > 0 && (!d || !g || !hbar || !accept))
        return fail(KVFIX_EINVAL, "%s: d, g, hbar and accept are required", fn);
    if (src.chunks > 0 && src.layers > 0) {
        if (!workspace || workspace_bytes < anchor_gate_workspace_bytes(src, anchors, src.tokens))
            return fail(KVFIX_EINVAL, "%s: workspace smaller than kvfix_anchor_gate_workspace_bytes(src, anchors, tokens)", fn);
        if (!aligned16(workspace)) return fail(KVFIX_EINVAL, "%s: workspace not 16-byte aligned", fn);
    }
    AnchorGateOut gate;
    gate.k = prefix;
    gate.T = temperature;
    gate.tau = tau;
    gate.d = d;
    gate.g = g;
    gate.hbar = hbar;
    gate.accept = accept;
    gate.workspace = workspace;
    return anchor_correct_impl(fn, k_src, v_src, src, a_c_k, b_ct_k, a_c_v, b_ct_v, a_d_k, b_dt_k, a_d_v, b_dt_v,
                               anchors, rank, temperature, delta, rope_base, nullptr, w_k, w_v, k_out, v_out, out,
                               stream, &gate);
}

// p / q rounded to the nearest integer, halves to even (p >= 0, q > 0).
static long long round_half_even(long long p, long long q) {
    long long f = p / q, r = p - f * q;
    if (2 * r > q || (2 * r == q && (f & 1))) ++f;
    return f;
}

kvfix_status kvfix_repair_layout(const double* scores, int32_t units, int32_t tokens, int32_t layout,
                                 int32_t chunk_tokens, int32_t budget_num, int32_t budget_den, double tau,
                                 int32_t skip_rule, int32_t* idx, int32_t max_rows, int32_t* counts,
                                 void* stream) {
    const char* fn = "kvfix_repair_layout";
    if (units < 0 || units > 65535) return fail(KVFIX_EINVAL, "%s: units must be in [0, 65535]", fn);
    if (tokens < 1 || tokens > 16384) return fail(KVFIX_EINVAL, "%s: tokens must be in [1, 16384]", fn);
    if (layout < 0 || layout > 2) return fail(KVFIX_EINVAL, "%s: unknown layout %d", fn, layout);
    if (layout == 1 && chunk_tokens < 1) return fail(KVFIX_EINVAL, "%s: chunk_tokens must be >= 1", fn);
    if (budget_den < 1 || budget_num < 0 || budget_num > budget_den)
        return fail(KVFIX_EINVAL, "%s: the budget must be a fraction in [0, 1]", fn);
    if (!isfinite(tau)) return fail(KVFIX_EINVAL, "%s: tau must be finite", fn);
    if (units > 0 && (!scores || !idx || !counts)) return fail(KVFIX_EINVAL, "%s: scores, idx and counts are required", fn);
    const long long n = tokens;
    int k = 0, c = 0, skipped = 0;
    long long need;
    if (layout == 1) {
        const long long B = chunk_tokens, nch = (n + B - 1) / B;
        skipped = skip_rule && (n < 2 * B || (long long)budget_num * n < (long long)budget_den * B);
        long long cc = round_half_even((long long)budget_num * n, (long long)budget_den * B);
        if (cc < 1) cc = 1;
        if (cc > nch) cc = nch;
        c = (int)cc;
        need = skipped ? 0 : (cc * B < n ? cc * B : n);
    } else {
        k = (int)round_half_even((long long)budget_num * n, budget_den);
        need = k;
    }
    if (max_rows < need || max_rows < 1)
        return fail(KVFIX_EINVAL, "%s: max_rows %d is below the layout's %lld rows", fn, max_rows, need);
    return launched(launch_repair_layout(scores, units, tokens, layout, chunk_tokens, k, c, skipped, tau, idx,
                                         max_rows, counts, (cudaStream_t)stream),
                    fn);
}

kvfix_status kvfix_repair_rows(kvfix_bf16* k_io, kvfix_bf16* v_io, kvfix_kv_desc desc, const kvfix_bf16* k_fresh,
                               const kvfix_bf16* v_fresh, kvfix_kv_desc fresh_desc, const int32_t* idx,
                               int32_t max_rows, const int32_t* counts, void* stream) {
    const char* fn = "kvfix_repair_rows";
    kvfix_status st;
    if ((k_io == nullptr) != (k_fresh == nullptr) || (v_io == nullptr) != (v_fresh == nullptr))
        return fail(KVFIX_EINVAL, "%s: each plane needs both its io and its fresh pointer, or neither", fn);
    if (k_io && (st = check_plane(k_io, desc, "kvfix_repair_rows: k_io")) != KVFIX_OK) return st;
    if (v_io && (st = check_plane(v_io, desc, "kvfix_repair_rows: v_io")) != KVFIX_OK) return st;
    if (k_fresh && (st = check_plane(k_fresh, fresh_desc, "kvfix_repair_rows: k_fresh")) != KVFIX_OK) return st;
    if (v_fresh && (st = check_plane(v_fresh, fresh_desc, "kvfix_repair_rows: v_fresh")) != KVFIX_OK) return st;
    if (!same_shape(desc, fresh_desc) || desc.chunks != fresh_desc.chunks)
        return fail(KVFIX_EINVAL, "%s: fresh planes must have the shape of desc", fn);
    if (max_rows < 0) return fail(KVFIX_EINVAL, "%s: negative max_rows", fn);
    if (max_rows > 0 && desc.chunks > 0 && (!idx || !counts)) return fail(KVFIX_EINVAL, "%s: idx and counts are required", fn);
    if (desc.layers > 65535 || desc.chunks > 65535) return fail(KVFIX_EINVAL, "%s: too many layers or chunks", fn);
    if ((k_io && (overlaps(k_io, desc, k_fresh, fresh_desc) || (v_fresh && overlaps(k_io, desc, v_fresh, fresh_desc)))) ||
        (v_io && (overlaps(v_io, desc, v_fresh, fresh_desc) || (k_fresh && overlaps(v_io, desc, k_fresh, fresh_desc)))) ||
        (k_io && v_io && overlaps(k_io, desc, v_io, desc)))
        return fail(KVFIX_EINVAL, "%s: planes overlap", fn);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (k_io && (e = launch_row_repair(k_io, desc, k_fresh, fresh_desc, idx, max_rows, s, counts)) != cudaSuccess)
        return cuda_fail(e, fn);
    if (v_io && (e = launch_row_repair(v_io, desc, v_fresh, fresh_desc, idx, max_rows, s, counts)) != cudaSuccess)
        return cuda_fail(e, fn);
    return KVFIX_OK;
}

kvfix_status kvfix_master_select(const float* d_k, const float* d_v, int32_t agents, int32_t units_per_agent,
                                 int32_t tokens, double* totals, int32_t* master, void* stream) {
    const char* fn = "kvfix_master_select";
    if (agents < 0 || agents > 65535 || units_per_agent < 1 || tokens < 1)
        return fail(KVFIX_EINVAL, "%s: agents in [0, 65535], units_per_agent and tokens >= 1", fn);
    if (agents > 0 && ((!d_k && !d_v) || !totals || !master))
        return fail(KVFIX_EINVAL, "%s: a score plane, totals and master are required", fn);
    return launched(launch_master_select(d_k, d_v, agents, units_per_agent, tokens, totals, master,
                                         (cudaStream_t)stream),
                    fn);
}

kvfix_status kvfix_diff_encode_split(const kvfix_bf16* master_k, const kvfix_bf16* master_v, kvfix_kv_desc master,
                                     const kvfix_bf16* sib_k, const kvfix_bf16* sib_v, kvfix_kv_desc sib,
                                     int32_t block_tokens, uint32_t* mask_k, uint32_t* mask_v, int64_t* offsets_k,
                                     int64_t* offsets_v, kvfix_bf16* payload_k, kvfix_bf16* payload_v,
                                     int64_t capacity_k, int64_t capacity_v, int64_t* h_entries, void* stream) {
    const char* fn = "kvfix_diff_encode_split";
    kvfix_status st;
    if ((st = check_plane(master_k, master, "kvfix_diff_encode_split: master_k")) != KVFIX_OK) return st;
    if ((st = check_plane(master_v, master, "kvfix_diff_encode_split: master_v")) != KVFIX_OK) return st;
    if ((st = check_plane(sib_k, sib, "kvfix_diff_encode_split: sib_k")) != KVFIX_OK) return st;
    if ((st = check_plane(sib_v, sib, "kvfix_diff_encode_split: sib_v")) != KVFIX_OK) return st;
    if (master.chunks != 1) return fail(KVFIX_EINVAL, "%s: master.chunks must be 1", fn);
    if (!same_shape(master, sib)) return fail(KVFIX_EINVAL, "%s: master and sibling shapes differ", fn);
    if (block_tokens < 1 || master.tokens % block_tokens)
        return fail(KVFIX_EINVAL, "%s: block_tokens must divide tokens", fn);
    if (!mask_k || !mask_v || !offsets_k || !offsets_v)
        return fail(KVFIX_EINVAL, "%s: both masks and both offset arrays are required", fn);
    if (capacity_k < 0 || capacity_v < 0) return fail(KVFIX_EINVAL, "%s: negative capacity", fn);
    if ((capacity_k > 0 && (!payload_k || !aligned16(payload_k))) || (capacity_v > 0 && (!payload_v || !aligned16(payload_v))))
        return fail(KVFIX_EINVAL, "%s: payloads must be 16-byte aligned device pointers", fn);
    const long long per_sibling = (long long)master.layers * (master.tokens / block_tokens);
    const long long entries = per_sibling * sib.chunks;
    if (entries >= (1ll << 31)) return fail(KVFIX_EINVAL, "%s: too many entries", fn);
    if (sib.chunks > 65535 || master.layers > 65535) return fail(KVFIX_EINVAL, "%s: at most 65535 siblings and layers", fn);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t mbytes = sizeof(uint32_t) * (size_t)((entries + 31) / 32);
    cudaError_t e;
    if ((e = cudaMemsetAsync(mask_k, 0, mbytes, s)) != cudaSuccess || (e = cudaMemsetAsync(mask_v, 0, mbytes, s)) != cudaSuccess)
        return cuda_fail(e, fn);
    if ((e = launch_diff_mask(master_k, master_v, master, sib_k, sib_v, sib, block_tokens, mask_k, s, mask_v)) != cudaSuccess)
        return cuda_fail(e, fn);
    if ((e = launch_diff_scan(mask_k, sib.chunks, per_sibling, offsets_k, s)) != cudaSuccess) return cuda_fail(e, fn);
    if ((e = launch_diff_scan(mask_v, sib.chunks, per_sibling, offsets_v, s)) != cudaSuccess) return cuda_fail(e, fn);
    if (h_entries) {
        int64_t tot[2] = {0, 0};
        if ((e = cudaMemcpyAsync(&tot[0], offsets_k + entries, sizeof(int64_t), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
            (e = cudaMemcpyAsync(&tot[1], offsets_v + entries, sizeof(int64_t), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e, fn);
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, fn);
        h_entries[0] = tot[0];
        h_entries[1] = tot[1];
        if (tot[0] > capacity_k || tot[1] > capacity_v)
            return fail(KVFIX_ENOSPACE, "%s: %lld + %lld entries needed, capacity %lld + %lld", fn, (long long)tot[0],
                        (long long)tot[1], (long long)capacity_k, (long long)capacity_v);
    }
    if (capacity_k > 0 &&
        (e = launch_diff_pack(sib_k, sib_v, sib, block_tokens, mask_k, offsets_k, payload_k, capacity_k, s, 1)) != cudaSuccess)
        return cuda_fail(e, fn);
    if (capacity_v > 0 &&
        (e = launch_diff_pack(sib_k, sib_v, sib, block_tokens, mask_v, offsets_v, payload_v, capacity_v, s, 2)) != cudaSuccess)
        return cuda_fail(e, fn);
    return KVFIX_OK;
}

kvfix_status kvfix_diff_gather_split(const kvfix_bf16* master_k, const kvfix_bf16* master_v, kvfix_kv_desc master,
                                     const uint32_t* mask_k, const uint32_t* mask_v, const int64_t* offsets_k,
                                     const int64_t* offsets_v, const kvfix_bf16* payload_k,
                                     const kvfix_bf16* payload_v, int64_t entries_k, int64_t entries_v,
                                     int32_t siblings, int32_t block_tokens, kvfix_bf16* out_k, kvfix_bf16* out_v,
                                     kvfix_kv_desc out, void* stream) {
    const char* fn = "kvfix_diff_gather_split";
    kvfix_status st;
    if ((st = check_plane(master_k, master, "kvfix_diff_gather_split: master_k")) != KVFIX_OK) return st;
    if ((st = check_plane(master_v, master, "kvfix_diff_gather_split: master_v")) != KVFIX_OK) return st;
    if ((st = check_plane(out_k, out, "kvfix_diff_gather_split: out_k")) != KVFIX_OK) return st;
    if ((st = check_plane(out_v, out, "kvfix_diff_gather_split: out_v")) != KVFIX_OK) return st;
    if (master.chunks != 1) return fail(KVFIX_EINVAL, "%s: master.chunks must be 1", fn);
    if (!same_shape(master, out) || out.chunks != siblings)
        return fail(KVFIX_EINVAL, "%s: out must have `siblings` chunks of the master's shape", fn);
    if (block_tokens < 1 || master.tokens % block_tokens)
        return fail(KVFIX_EINVAL, "%s: block_tokens must divide tokens", fn);
    if (siblings < 0 || siblings > 65535 || master.layers > 65535)
        return fail(KVFIX_EINVAL, "%s: siblings and layers must be <= 65535", fn);
    if (!mask_k || !mask_v || !offsets_k || !offsets_v)
        return fail(KVFIX_EINVAL, "%s: both masks and both offset arrays are required", fn);
    if (entries_k < 0 || entries_v < 0) return fail(KVFIX_EINVAL, "%s: negative payload entries", fn);
    if ((entries_k > 0 && (!payload_k || !aligned16(payload_k))) || (entries_v > 0 && (!payload_v || !aligned16(payload_v))))
        return fail(KVFIX_EINVAL, "%s: payloads must be 16-byte aligned device pointers", fn);
    if (overlaps(out_k, out, master_k, master) || overlaps(out_v, out, master_v, master) ||
        overlaps(out_k, out, out_v, out))
        return fail(KVFIX_EINVAL, "%s: outputs overlap the master or each other", fn);
    return launched(launch_diff_gather(master_k, master_v, master, mask_k, offsets_k, payload_k, entries_k, siblings,
                                       block_tokens, out_k, out_v, out, (cudaStream_t)stream, mask_v, offsets_v,
                                       payload_v, entries_v),
                    fn);
}

kvfix_status kvfix_selftest_wait(int64_t limit_cycles, const int32_t* flag, void* stream) {
    if (limit_cycles < 1 || limit_cycles > 4000000000ll)
        return fail(KVFIX_EINVAL, "kvfix_selftest_wait: limit_cycles must be in [1, 4e9]");
    return launched(launch_selftest_wait(limit_cycles, flag, (cudaStream_t)stream), "kvfix_selftest_wait");
}

}  // extern "C"
