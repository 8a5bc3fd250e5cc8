// noalloc.cu -- kvfix_draft_rank_noalloc: the draft-rank call with its scratch in a
// fixed device buffer that the library owns, for callers that cannot allocate.
//
// kvfix_draft_rank needs a workspace (attention logits and softmax statistics) that
// the caller normally allocates.  Some callers cannot: a serving engine that hands
// nearly all of HBM to its own KV-block pool at start-up (a later cudaMalloc fails or
// fragments that pool), or a latency-critical path that must not pay the device-wide
// synchronisation a cudaMalloc/cudaFree can imply.  This entry point takes the same
// arguments minus the workspace and uses the file-scope buffer below instead.  It
// calls no cudaMalloc, no cudaFree and no allocating library routine.
//
// Costs and rules of the shared buffer:
//  - the buffer (KVFIX_DRAFT_NOALLOC_SCRATCH_BYTES) is reserved on every GPU that
//    loads this library and stays reserved until the process exits;
//  - every call on a device uses the same buffer, so calls whose kernels overlap on
//    the GPU (different streams without ordering between them) race and give wrong
//    results; order them on one stream or with events;
//  - the buffer keeps the previous call's contents; nothing in it has to start at
//    zero, because every word a call reads was written earlier in that same call;
//  - the first call on a device looks up the buffer's device address (with that device
//    current), so make that first call before any stream capture begins.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "internal.h"

namespace kvfix {

static __device__ __align__(256) unsigned char g_draft_scratch[KVFIX_DRAFT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mutex;
static void* g_scratch_addr[kMaxDevices];

// Device address of this device's copy of the buffer (looked up once per device).
static kvfix_status scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "kvfix_draft_rank_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return fail(KVFIX_EINVAL, "kvfix_draft_rank_noalloc: device index %d not supported", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_draft_scratch);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e,
                             "kvfix_draft_rank_noalloc: cudaGetSymbolAddress of the scratch buffer");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KVFIX_OK;
}

}  // namespace kvfix

using namespace kvfix;

extern "C" kvfix_status kvfix_draft_rank_noalloc(const kvfix_bf16* k, kvfix_kv_desc desc,
                                                 const kvfix_bf16* q, int32_t draft_steps,
                                                 int32_t q_heads, int32_t layer_begin,
                                                 int32_t k_rows, int32_t* idx, double* scores,
                                                 const kvfix_bf16* k_fresh,
                                                 const kvfix_bf16* v_fresh,
                                                 kvfix_kv_desc fresh_desc, kvfix_bf16* k_io,
                                                 kvfix_bf16* v_io, void* stream) {
    if (layer_begin < 0 || layer_begin > desc.layers || desc.chunks < 0 || desc.layers < 0 ||
        desc.tokens < 0 || desc.kv_heads < 1)
        return fail(KVFIX_EINVAL, "kvfix_draft_rank_noalloc: bad descriptor or layer_begin");
    const size_t need = kvfix_draft_rank_workspace_bytes(desc, layer_begin);
    const size_t have = (size_t)KVFIX_DRAFT_NOALLOC_SCRATCH_BYTES;
    if (need > have)
        return fail(KVFIX_EINVAL,
                    "kvfix_draft_rank_noalloc: this problem needs %zu bytes of scratch but the "
                    "fixed buffer holds %zu; split it into smaller calls or use kvfix_draft_rank "
                    "with a caller-allocated workspace",
                    need, have);
    void* ws = nullptr;
    kvfix_status st = scratch_for_current_device(&ws);
    if (st != KVFIX_OK) return st;
    st = kvfix_draft_rank(k, desc, q, draft_steps, q_heads, layer_begin, k_rows, idx, scores, k_fresh,
                          v_fresh, fresh_desc, k_io, v_io, ws, have, stream);
    if (st != KVFIX_OK) {  // name this entry point in the message of the inner call's error
        char inner[400];
        snprintf(inner, sizeof inner, "%s", kvfix_last_error());
        return fail(st, "kvfix_draft_rank_noalloc: %s", inner);
    }
    return KVFIX_OK;
}
