/*
 * kvfix.h -- C ABI of libkvfix, the repair path for reused KV-cache chunks on one
 * NVIDIA GB300 (sm_103a).
 *
 * The library re-aligns, scores, selects, corrects and stores KV caches that one
 * agent reuses from another context.  Every call enqueues hand-written CUDA kernels
 * on the caller's stream; nothing runs on the host but argument checks.
 *
 * Conventions shared by every call
 * --------------------------------
 * - bf16 tensors are passed as `kvfix_bf16*`: raw IEEE bfloat16 bit patterns.
 * - All tensor pointers are DEVICE pointers unless the name starts with `h_`.
 * - A KV plane (the keys or the values of a cache) is described by kvfix_kv_desc:
 *   element (c, l, t, h, e) -- chunk, layer, token, KV head, head dim -- lives at
 *       c*stride_chunk + l*stride_layer + t*stride_token + h*head_dim + e
 *   (strides in elements).  The heads of one token are contiguous (one token row is
 *   kv_heads*head_dim elements).  head_dim must be a multiple of 16 in [16, 256]; the
 *   base pointer must be 16-byte aligned and every stride a non-negative multiple of
 *   8 elements, so that rows move as 16-byte vectors.
 * - `stream` is a cudaStream_t cast to void* (NULL = the legacy default stream).
 * - Ownership: the caller owns every buffer.  The library keeps no per-call state
 *   and allocates no device memory; calls that need scratch take a workspace
 *   buffer whose size a companion *_workspace_bytes() query returns.
 * - Errors: arguments are checked on the host before anything is launched; a bad
 *   argument returns KVFIX_EINVAL and launches nothing.  A launch failure returns
 *   KVFIX_ECUDA.  kvfix_last_error() gives the message of the last non-OK status of
 *   the calling thread.  Conditions only the GPU can see (an index in caller data
 *   out of range, a payload overflow) set a device status word instead; the kernels
 *   then skip the offending access.  kvfix_check_status() reads and clears it.
 * - Calls are asynchronous: a KVFIX_OK return means "enqueued".
 * - Outputs never alias inputs, except where a call says so.
 *
 * Citations name the page and section that define each operation:
 *   [KVCMAS]  KVCMAS: Efficient KV cache Correction for Shared Context in Multi-Agent Systems
 *   [AKS]     AgentKVShift: Correcting Reused KV (review)
 *   [TD]      TokenDance: Scaling Multi-Agent LLM Serving via Collective KV Cache Sharing (summary)
 *   [BCR]     Budgeted Cache Repair for Cross-Context KV-Cache Reuse
 */
#ifndef KVFIX_H
#define KVFIX_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVFIX_API __attribute__((visibility("default")))
#else
#define KVFIX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvfix_bf16;

typedef enum {
    KVFIX_OK = 0,
    KVFIX_EINVAL = 1,   /* bad argument; nothing was launched */
    KVFIX_ENOSPACE = 2, /* diff payload capacity too small (see kvfix_diff_encode) */
    KVFIX_ECUDA = 3,    /* a CUDA runtime call or launch failed */
    KVFIX_ETIMEOUT = 4, /* a bounded device-side wait gave up */
    KVFIX_EDEVICE = 5   /* the device flagged bad caller data (index out of range) */
} kvfix_status;

typedef struct {
    int32_t chunks;
    int32_t layers;
    int32_t tokens;
    int32_t kv_heads;
    int32_t head_dim;
    int64_t stride_chunk;
    int64_t stride_layer;
    int64_t stride_token;
} kvfix_kv_desc;

/* Library version, major*10000 + minor*100 + patch. */
KVFIX_API int kvfix_version(void);

/* Message of the calling thread's last non-OK status ("" if none).  The pointer
 * stays valid until the thread's next kvfix call. */
KVFIX_API const char* kvfix_last_error(void);

/* Synchronise `stream`, then read and clear the device status word.
 * Returns KVFIX_OK, KVFIX_EDEVICE (an index out of range was skipped),
 * KVFIX_ENOSPACE (a payload write was skipped), KVFIX_ETIMEOUT or KVFIX_ECUDA. */
KVFIX_API kvfix_status kvfix_check_status(void* stream);

/*
 * kvfix_rerope -- re-align cached keys to new positions with rotary embeddings.
 * [KVCMAS] section 2.2 and App. A.3 (keys are re-aligned to their target positions,
 * values are not rotated); [TD] section 4.4, Algorithm 1 (RoPERecover(P_old, P_new));
 * [BCR] App. A (one scalar position shift per reused segment).
 *
 * With rotate-half RoPE, theta_i = rope_base^(-2i/D) for i < D/2 and dimension i
 * paired with i + D/2, a key encoded at position p and moved to p + delta is rotated
 * once more by the angle delta*theta_i:
 *     y_i       = x_i cos(delta theta_i) - x_{i+D/2} sin(delta theta_i)
 *     y_{i+D/2} = x_{i+D/2} cos(delta theta_i) + x_i sin(delta theta_i)
 * k_in, k_out : one KV plane each, described by in_desc / out_desc (same shape; k_out
 *               may be k_in itself with the same descriptor, for an in-place update).
 * delta       : device int32[in_desc.chunks], the shift of each chunk (any sign).
 * Arithmetic: angles reduced in double, cos/sin and the rotation in float, output
 * rounded to nearest-even bf16.  delta = 0 reproduces the input bit for bit.
 */
KVFIX_API kvfix_status kvfix_rerope(const kvfix_bf16* k_in, kvfix_kv_desc in_desc, kvfix_bf16* k_out,
                                    kvfix_kv_desc out_desc, const int32_t* delta, double rope_base,
                                    void* stream);

/*
 * kvfix_score_topk -- check-layer divergence and probe selection.
 * [AKS] "Core idea and method", steps 1-2 and the displayed b, d and w equations;
 * [TD] section 4.2 (one batched rotation and one batched check-layer comparison for
 * all requests of a round).
 *
 * Units: unit u = a*R + r pairs agent a (of `agents`) with reused chunk r (of
 * R = reuse.chunks).  For every unit and token j of the check layer:
 *     d_k[u][j] = || k_fresh[u][j] - rerope(k_reuse[r][j], delta[u]) ||_2
 *     d_v[u][j] = || v_fresh[u][j] - v_reuse[r][j] ||_2
 * where the norm runs over the whole token row (all KV heads).  Then, for each plane,
 * the b tokens with the largest d (ties to the lower index; d compared as float) are
 * the probes: idx_*[u][0..b-1] in ascending order, bit j of mask_*[u] set for each
 * (word j/32, bit j%32), w_*[u][j] = min(d[u][j], 1).  mask_union = mask_k | mask_v.
 *
 * k_reuse, v_reuse : check-layer views, `reuse` (layers == 1), R chunks.
 * k_fresh, v_fresh : check-layer views, `fresh` (layers == 1, chunks == agents*R,
 *                    same tokens/heads/head_dim as `reuse`).
 * delta            : device int32[agents*R].
 * b                : 0 <= b <= tokens (b = ceil(r n) for probe ratio r).
 * d_k, d_v, w_k, w_v : device float[agents*R][tokens], required.
 * idx_k, idx_v     : device int32[agents*R][b], required when b > 0.
 * mask_k, mask_v, mask_union : device uint32[agents*R][ceil(tokens/32)], optional.
 * Limits: tokens <= 65536.  All agents of a round are handled by one set of launches;
 * each reused check-layer row is read once for all agents.
 */
KVFIX_API kvfix_status kvfix_score_topk(const kvfix_bf16* k_reuse, const kvfix_bf16* v_reuse,
                              kvfix_kv_desc reuse, const kvfix_bf16* k_fresh,
                              const kvfix_bf16* v_fresh, kvfix_kv_desc fresh, int32_t agents,
                              const int32_t* delta, double rope_base, int32_t b, float* d_k,
                              float* d_v, float* w_k, float* w_v, int32_t* idx_k, int32_t* idx_v,
                              uint32_t* mask_k, uint32_t* mask_v, uint32_t* mask_union,
                              void* stream);

/*
 * kvfix_mean_correct -- probe-mean residual correction of every layer.
 * [AKS] "Core idea and method", steps 3-4 and the displayed mu-hat and K_corr
 * equations; [TD] section 4.2 (only the per-request refresh differs between the
 * requests of a group).
 *
 * For unit u = a*R + r, layer l, plane P in {K, V} with probe list S = idx_P[u][0..b-1]
 * and weights w_P[u]:
 *     mu_P[u][l][h*D+e] = (1/b) sum_{i<b} (fresh_P[u][l][S_i][h][e] - rot(reuse_P[r][l][S_i][h])[e])
 *     out_P[u][l][j]    = fresh_P[u][l][j]                              if j in S (bit copy)
 *                       = bf16(rot(reuse_P[r][l][j]) + w_P[u][j] * mu_P[u][l])   otherwise
 * rot is the re-rope by delta[u] for keys and the identity for values; b == 0 gives
 * mu = 0 and out = bf16(rot(reuse)).  The sum runs in a fixed order (probe i goes to
 * partial sum i mod 32; partial sums are added in order), so a round of N agents in
 * one call and N one-agent calls give the same bits.
 *
 * reuse, fresh, out : plane descriptors; reuse has R chunks, fresh and out agents*R,
 *                     all with the same layers/tokens/heads/head_dim.
 * k_* / v_*         : pass all NULL for a plane to skip it.
 * idx_k, idx_v      : device int32[agents*R][b] (ascending not required; each entry
 *                     must lie in [0, tokens) -- others are skipped and flagged).
 * w_k, w_v          : device float[agents*R][tokens].
 * mu_k, mu_v        : device float[agents*R][layers][kv_heads*head_dim], written (and
 *                     read back by the call's second kernel); must not overlap w or out.
 * Each reused row is read once for all agents of the call.
 */
KVFIX_API kvfix_status kvfix_mean_correct(const kvfix_bf16* k_reuse, const kvfix_bf16* v_reuse,
                                kvfix_kv_desc reuse, const kvfix_bf16* k_fresh,
                                const kvfix_bf16* v_fresh, kvfix_kv_desc fresh, kvfix_bf16* k_out,
                                kvfix_bf16* v_out, kvfix_kv_desc out, int32_t agents,
                                const int32_t* delta, double rope_base, const int32_t* idx_k,
                                const int32_t* idx_v, int32_t b, const float* w_k,
                                const float* w_v, float* mu_k, float* mu_v, void* stream);

/*
 * kvfix_lowrank_apply -- add a rank-r factorised delta to a KV plane.
 * [KVCMAS] Eq. 4 (corrected cache = reference + estimated delta), Eq. 7 (a delta
 * stored as A B, A of size rows x r, B of size r x D), Eq. 8 with a single anchor.
 *
 *     out[c][l][j][h][e] = bf16( x[c][l][j][h][e] + sum_{k<r} A[c][l][h][j][k] B[c][l][h][k][e] )
 * x, out : one KV plane each, described by desc / out_desc (same shape); out may be x
 *          itself with the same descriptor (in place).
 * A      : device bf16[chunks][layers][kv_heads][tokens][rank], contiguous.
 * B      : device bf16[chunks][layers][kv_heads][rank][head_dim], contiguous.
 * rank   : 16, 32 or 64.  head_dim must be 64 or 128.
 * Arithmetic: bf16 products on the tensor cores (tcgen05, accumulator in tensor memory)
 * with float accumulation, then the add in float and one rounding to bf16.
 */
KVFIX_API kvfix_status kvfix_lowrank_apply(const kvfix_bf16* x, kvfix_kv_desc desc, const kvfix_bf16* A,
                                           const kvfix_bf16* B, int32_t rank, kvfix_bf16* out,
                                           kvfix_kv_desc out_desc, void* stream);

/*
 * kvfix_draft_rank -- rank cached rows by the attention mass of draft queries, keep
 * the best k_rows, and optionally repair them.
 * [BCR] section 3 ("The repair": the row score a_j), App. B Algorithm 2 (draft
 * scoring with grouped-query keys expanded to query heads) and Algorithm 1 (the
 * selected rows' K and V overwritten with exact ones); [KVCMAS] Eq. 3.
 *
 *     scores[c][j] = sum_{l >= layer_begin} sum_{t < draft_steps} sum_{h < q_heads}
 *                    softmax_j( q[c][l][t][h] . k[c][l][j][h / (q_heads/kv_heads)] / sqrt(D) )
 * (summed over (t, h); the ranking equals the mean's).  idx[c] = the k_rows rows with
 * the largest score (ties to the lower index), ascending.
 * If k_io / v_io are non-NULL, then for every layer and KV head, rows idx[c] of k_io /
 * v_io are overwritten with the same rows of k_fresh / v_fresh.  k_io may be the
 * scored buffer `k` itself (the overwrite runs after scoring, in stream order).
 *
 * k              : the assembled keys, `desc` (heads = kv_heads).
 * q              : device bf16[chunks][layers][draft_steps][q_heads][head_dim], contiguous.
 * idx            : device int32[chunks][k_rows]; scores: device double[chunks][tokens].
 * k_fresh, v_fresh, k_io, v_io : planes described by `fresh_desc` / `desc`, or NULL.
 * workspace      : device buffer of kvfix_draft_rank_workspace_bytes(desc, layer_begin)
 *                  bytes (16-byte aligned), contents irrelevant on entry.
 * Limits: q_heads a multiple of kv_heads, q_heads/kv_heads * draft_steps <= 16,
 * head_dim 64 or 128, tokens <= 16384 per chunk, chunks * (layers - layer_begin) *
 * kv_heads <= 65535, 0 <= k_rows <= tokens.
 * Arithmetic: the logits are a bf16 tensor-core contraction (tcgen05) with float
 * accumulation kept in tensor memory; softmax statistics in float; per-unit masses in
 * float, summed over the units of a chunk in a fixed order (layer-major, then head) as
 * a compensated float pair (running sum plus its accumulated rounding errors, about 48
 * significant bits), returned as the double hi + lo.
 */
KVFIX_API size_t kvfix_draft_rank_workspace_bytes(kvfix_kv_desc desc, int32_t layer_begin);
KVFIX_API kvfix_status kvfix_draft_rank(const kvfix_bf16* k, kvfix_kv_desc desc, const kvfix_bf16* q,
                              int32_t draft_steps, int32_t q_heads, int32_t layer_begin,
                              int32_t k_rows, int32_t* idx, double* scores,
                              const kvfix_bf16* k_fresh, const kvfix_bf16* v_fresh,
                              kvfix_kv_desc fresh_desc, kvfix_bf16* k_io, kvfix_bf16* v_io,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvfix_lowrank_draft -- kvfix_lowrank_apply of the key plane and kvfix_draft_rank of the
 * corrected keys in one pass: each corrected key tile is scored while it is still on chip,
 * so the corrected keys are read from memory by neither step.
 * [KVCMAS] Eq. 4, 7, 8 (corrected keys = reference keys + A B); [BCR] section 3 ("The
 * repair": rows ranked by the draft queries' attention mass over the predicted keys) and
 * App. B Algorithms 1 and 2.
 *
 * Computes exactly what these calls compute, in this order:
 *     kvfix_lowrank_apply(x, desc, A, B, rank, out, out_desc)
 *     kvfix_draft_rank(out, out_desc, q, draft_steps, q_heads, layer_begin, k_rows, idx,
 *                      scores, k_fresh, v_fresh, fresh_desc, k_fresh ? out : NULL, v_io)
 * with the same bits: out, idx and scores equal the two-call sequence's.  The value
 * plane's low-rank delta is a separate kvfix_lowrank_apply (give its output as v_io to
 * repair its rows here).
 * Arguments are those of the two calls: x/out/A/B/rank as for kvfix_lowrank_apply (out may
 * be x itself, in place); q, draft_steps, q_heads, layer_begin, k_rows, idx and scores as
 * for kvfix_draft_rank.  workspace: device buffer of
 * kvfix_lowrank_draft_workspace_bytes(desc, layer_begin) bytes (16-byte aligned; the
 * draft workspace plus a fixed 132 KB exchange area), contents irrelevant on entry.  k_fresh (optional): the selected rows of out are overwritten with it;
 * v_fresh with v_io (optional): the selected rows of v_io (shaped like out) are
 * overwritten with it.  Limits: head_dim 64 or 128, rank 16/32/64, tokens <= 16384,
 * (q_heads/kv_heads)*draft_steps <= 16.
 * Runs as one persistent cooperative kernel (one CTA per SM, all of its tensor memory;
 * it fails with KVFIX_ECUDA if the device cannot hold one CTA on each SM it uses), then
 * the per-key sums, the top-k and the row repair.
 */
KVFIX_API size_t kvfix_lowrank_draft_workspace_bytes(kvfix_kv_desc desc, int32_t layer_begin);
KVFIX_API kvfix_status kvfix_lowrank_draft(const kvfix_bf16* x, kvfix_kv_desc desc, const kvfix_bf16* A,
                                           const kvfix_bf16* B, int32_t rank, kvfix_bf16* out,
                                           kvfix_kv_desc out_desc, const kvfix_bf16* q, int32_t draft_steps,
                                           int32_t q_heads, int32_t layer_begin, int32_t k_rows, int32_t* idx,
                                           double* scores, const kvfix_bf16* k_fresh, const kvfix_bf16* v_fresh,
                                           kvfix_kv_desc fresh_desc, kvfix_bf16* v_io, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * kvfix_draft_rank_noalloc -- kvfix_draft_rank for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a service of this library only.
 *
 * Who needs it: a serving engine that gives nearly all of HBM to its own KV-block
 * pool at start-up (a later cudaMalloc fails or fragments the pool), or a
 * latency-critical path that must not pay the device-wide synchronisation a
 * cudaMalloc/cudaFree can imply.  Same arguments and results as kvfix_draft_rank,
 * without the workspace: the scratch lives in a fixed buffer of
 * KVFIX_DRAFT_NOALLOC_SCRATCH_BYTES that the library reserves on every GPU that loads
 * it, until the process exits.  The call allocates nothing.
 * - A problem that needs more scratch than the buffer holds
 *   (kvfix_draft_rank_workspace_bytes(desc, layer_begin) > the constant) returns
 *   KVFIX_EINVAL with a message and launches nothing.
 * - All calls on a device share the buffer: calls whose kernels overlap on the GPU
 *   race.  Order them (one stream, or events).
 * - The buffer keeps the last call's contents; nothing in it needs to start at zero.
 * - The first call on a device looks up the buffer's device address with that device
 *   current; make that first call before any stream capture begins.
 */
#define KVFIX_DRAFT_NOALLOC_SCRATCH_BYTES (64u << 20)
KVFIX_API kvfix_status kvfix_draft_rank_noalloc(const kvfix_bf16* k, kvfix_kv_desc desc,
                                                const kvfix_bf16* q, int32_t draft_steps,
                                                int32_t q_heads, int32_t layer_begin,
                                                int32_t k_rows, int32_t* idx, double* scores,
                                                const kvfix_bf16* k_fresh,
                                                const kvfix_bf16* v_fresh,
                                                kvfix_kv_desc fresh_desc, kvfix_bf16* k_io,
                                                kvfix_bf16* v_io, void* stream);

/*
 * kvfix_diff_encode -- store sibling caches as block-sparse diffs against a master.
 * [TD] section 4.3 (master-mirror layout, block-sparse K/V diff) and section 5 (a
 * mirror keeps the touched block indices and those blocks' K/V contents; one index
 * list shared by K and V).
 *
 * Entry i = (s*L + l)*nblk + blk covers tokens [bt*blk, bt*blk + bt) of layer l of
 * sibling s, all heads, both planes (nblk = tokens / bt).  It is dirty iff some bf16
 * word of K or V in it differs bitwise from the master's (so -0 differs from +0).
 *     mask    : device uint32[ceil(S*L*nblk/32)], bit i%32 of word i/32 = dirty
 *     offsets : device int64[S*L*nblk + 1], offsets[i] = dirty entries before i,
 *               offsets[S*L*nblk] = total
 *     payload : device bf16[capacity_entries][2][bt][kv_heads][head_dim]; dirty entry
 *               i is stored at offsets[i]: the sibling's K block, then its V block.
 * master_* : `master` (chunks == 1); sib_* : `sib` (chunks = S siblings, same shape).
 * h_entries: optional HOST pointer.  If given, the call synchronises the stream after
 *            the mask and offsets are built, stores the total there and returns
 *            KVFIX_ENOSPACE without writing the payload if it exceeds
 *            capacity_entries.  If NULL the call stays asynchronous and the device
 *            skips (and flags) entries beyond capacity_entries.
 * bt must divide tokens.
 */
KVFIX_API kvfix_status kvfix_diff_encode(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                               kvfix_kv_desc master, const kvfix_bf16* sib_k,
                               const kvfix_bf16* sib_v, kvfix_kv_desc sib, int32_t block_tokens,
                               uint32_t* mask, int64_t* offsets, kvfix_bf16* payload,
                               int64_t capacity_entries, int64_t* h_entries, void* stream);

/*
 * kvfix_diff_gather -- restore every sibling from the master and its diff.
 * [TD] section 4.4, Algorithm 1 (load the master block, overwrite the blocks the diff
 * touches with the diff's values); section 5 (paired K/V diff kernel).
 *
 *     out_P[s][l][block blk] = payload[offsets[i]].P   if mask bit i is set
 *                            = master_P[l][block blk]   otherwise
 * Each master block is read once for all siblings.
 * mask, offsets, payload : as written by kvfix_diff_encode.
 * payload_entries        : entries the payload buffer holds; a dirty entry whose offset
 *                          lies beyond it is not read (its block gets the master's
 *                          contents) and is flagged (KVFIX_ENOSPACE in kvfix_check_status).
 * out_k, out_v           : `out` (chunks = siblings, same shape as master).
 */
KVFIX_API kvfix_status kvfix_diff_gather(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                               kvfix_kv_desc master, const uint32_t* mask,
                               const int64_t* offsets, const kvfix_bf16* payload,
                               int64_t payload_entries, int32_t siblings, int32_t block_tokens,
                               kvfix_bf16* out_k, kvfix_bf16* out_v, kvfix_kv_desc out,
                               void* stream);

/*
 * kvfix_diff_restore -- fused restore of every sibling into a paged KV pool.
 * [TD] section 4.4, Algorithm 1 (per layer: load the master block, overwrite it where
 * the sibling's block-sparse diff touches it, re-align the keys from the old to the new
 * positions with RoPERecover, write the rows to the paged cache through the slot
 * mapping); section 5 (the restore is one fused kernel, no intermediate full copy).
 *
 * Re-alignment of sibling s is one rotary shift by delta[s] = P_new - P_old (as in
 * kvfix_rerope; values are not rotated).  Token t of sibling s is written, in every
 * layer, to pool row slot_mapping[s*tokens + t]:
 *     pool_k[l][slot] = rotate(delta[s], restored K row),  pool_v[l][slot] = restored V row
 * where the restored row is the payload's if the entry is dirty, else the master's.
 * A negative slot means the token is not restored; a slot >= pool.tokens is skipped
 * and flagged (KVFIX_EDEVICE in kvfix_check_status).  Pool rows no slot names are left
 * unchanged.  Slots must be distinct (two tokens naming one row race).
 * master_*, mask, offsets, payload, payload_entries, siblings, block_tokens: as for
 *                  kvfix_diff_gather.
 * delta          : device int32[siblings].
 * rope_base      : as for kvfix_rerope.
 * slot_mapping   : device int32[siblings][tokens].
 * pool_k, pool_v : `pool` -- chunks == 1, layers and heads x head_dim as the master's,
 *                  tokens = the pool's rows per layer; neither may overlap the master.
 * delta[s] = 0 copies sibling s's keys bit for bit.
 */
KVFIX_API kvfix_status kvfix_diff_restore(const kvfix_bf16* master_k, const kvfix_bf16* master_v,
                                kvfix_kv_desc master, const uint32_t* mask,
                                const int64_t* offsets, const kvfix_bf16* payload,
                                int64_t payload_entries, int32_t siblings, int32_t block_tokens,
                                const int32_t* delta, double rope_base,
                                const int32_t* slot_mapping, kvfix_bf16* pool_k,
                                kvfix_bf16* pool_v, kvfix_kv_desc pool, void* stream);

/*
 * Anchor-pool correction.  [KVCMAS] section 3.3 (each anchor keeps its base cache and its
 * delta correction as low-rank factors, Eq. 7; the correction is the weighted sum of the
 * anchors' deltas, Eq. 8, applied to the aligned source cache, Eq. 4) and App. A.3
 * (reliability gate, Eq. 9-11; token-wise weights; keys matched in canonical positions).
 *
 * Factor layout, per plane, for C segments (src.chunks), V anchors, L layers, n tokens,
 * F = kv_heads * head_dim features and rank r:
 *     A  : device bf16 [C][V][L][n][r]        (first factor, row t of the segment)
 *     Bt : device bf16 [C][V][L][F][r]        (second factor, stored transposed)
 * so that anchor v's state of layer l is A[c][v][l] * Bt[c][v][l]^T ([n x F]).
 * anchors: 1..16; rank: 16, 32 or 64 (the first-factor tiles of all anchors stay in
 * shared memory: ranks 16 and 32 take up to 16 anchors, rank 64 up to 8; the calls return
 * KVFIX_EINVAL for shapes that do not fit); F must be a multiple of 128.
 */

/* Bytes of device workspace kvfix_anchor_gate needs for `src`, `anchors` and `prefix`. */
KVFIX_API size_t kvfix_anchor_gate_workspace_bytes(kvfix_kv_desc src, int32_t anchors,
                                                   int32_t prefix);

/*
 * kvfix_anchor_gate -- [KVCMAS] App. A.3 "Reliability Gate", Eq. 9-11, per segment c:
 *     d_v  = ( sum_l || V_src^(l)[:k] - (A_v Bt_v^T)^(l)[:k] ||_F^2 )^(1/2)
 *     g_v  = softmax_v(-d_v / T),   Hbar = -sum_v g_v log2 g_v / log2 V
 *     accept = V >= 2 && Hbar <= tau
 * v_src      : `src`, the source value plane (chunks = segments).
 * a_c, b_ct  : base-state factors of the value plane (layout above).
 * prefix k   : 1..tokens; temperature T > 0.
 * d, g       : device double [C][V];  hbar : device double [C] (NaN if V < 2);
 * accept     : device int32 [C].  Distances are summed per 128-row tile in float and
 *              across tiles and layers in double, in a fixed order.
 * workspace  : device, at least kvfix_anchor_gate_workspace_bytes(), 16-byte aligned.
 */
KVFIX_API kvfix_status kvfix_anchor_gate(const kvfix_bf16* v_src, kvfix_kv_desc src,
                                         const kvfix_bf16* a_c, const kvfix_bf16* b_ct,
                                         int32_t anchors, int32_t rank, int32_t prefix,
                                         double temperature, double tau, double* d, double* g,
                                         double* hbar, int32_t* accept, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * kvfix_anchor_correct -- token-weighted anchor correction of both planes:
 *     m_v[t] = (1/F) sum_f | x[t][f] - (A_c,v Bt_c,v^T)[t][f] |   (x: keys in canonical positions)
 *     w[t]   = softmax_v(-m_v[t] / T)                            (per plane, layer, token)
 *     out[t] = Align(x[t]) + sum_v w_v[t] (A_d,v Bt_d,v^T)[t]     (bf16)
 * Align rotates keys by delta[c] (as kvfix_rerope) and leaves values unchanged.
 * k_src, v_src : `src` (chunks = segments); head_dim 64 or 128.
 * a_c_*, b_ct_*: base-state factors; a_d_*, b_dt_*: delta-correction factors (layout above).
 * delta        : device int32 [C]; rope_base as for kvfix_rerope.
 * accept       : optional device int32 [C] (e.g. kvfix_anchor_gate's): segments with 0 are
 *                skipped entirely (outputs and weights untouched).  NULL corrects all.
 * w_k, w_v     : device float [C][L][n][V], written with the token weights.
 * k_out, v_out : `out`, the shape of src; may be exactly src (in place), no other overlap.
 * The delta term is formed on the tensor cores from bf16(w_v * A_d,v) (the weight is
 * folded into the first factor, rounded once to bf16) with float accumulation.
 */
KVFIX_API kvfix_status kvfix_anchor_correct(
    const kvfix_bf16* k_src, const kvfix_bf16* v_src, kvfix_kv_desc src, const kvfix_bf16* a_c_k,
    const kvfix_bf16* b_ct_k, const kvfix_bf16* a_c_v, const kvfix_bf16* b_ct_v,
    const kvfix_bf16* a_d_k, const kvfix_bf16* b_dt_k, const kvfix_bf16* a_d_v,
    const kvfix_bf16* b_dt_v, int32_t anchors, int32_t rank, double temperature,
    const int32_t* delta, double rope_base, const int32_t* accept, float* w_k, float* w_v,
    kvfix_bf16* k_out, kvfix_bf16* v_out, kvfix_kv_desc out, void* stream);

/*
 * kvfix_repair_layout -- the rows a draft-scored repair recomputes, in one of the layouts
 * of [BCR] section 3 "The layouts", App. A.2 ("The policy", Table 8) and App. B
 * (Algorithms 1 and 2).  For each unit u of scores [units][tokens]
 * (e.g. kvfix_draft_rank's), with rho = budget_num / budget_den and rounding of halves
 * to even:
 *   KVFIX_LAYOUT_SINGLE: the round(rho n) rows with the largest scores;
 *   KVFIX_LAYOUT_CHUNK : chunk_tokens-token chunks (the last may be short), each scored by
 *                        the mean of its rows' scores (summed in index order, in double);
 *                        the max(1, round(rho n / chunk_tokens)) best chunks, all their
 *                        rows.  skip_rule != 0: no rows when n < 2 chunk_tokens or
 *                        rho n < chunk_tokens (Algorithm 1's skip rule);
 *   KVFIX_LAYOUT_GROW  : round(rho n) rows: the best unselected row seeds a span, which
 *                        takes the better of its two unselected neighbours (left on a tie)
 *                        while that one scores at least tau times the seed, until neither
 *                        does or the budget is spent; then the next seed.
 * Ties go to the lower index.  Scores must be finite.
 * idx      : device int32 [units][max_rows]: the rows, ascending, then -1.
 * counts   : device int32 [units]: rows chosen (the same for every unit except when the
 *            chunk layout's last, short chunk is chosen).
 * max_rows : at least the layout's largest count (KVFIX_EINVAL otherwise): round(rho n)
 *            for single and grow, (chunks chosen) * chunk_tokens (at most n) for chunk.
 * tokens   : 1..16384.
 */
typedef enum { KVFIX_LAYOUT_SINGLE = 0, KVFIX_LAYOUT_CHUNK = 1, KVFIX_LAYOUT_GROW = 2 } kvfix_layout;
KVFIX_API kvfix_status kvfix_repair_layout(const double* scores, int32_t units, int32_t tokens,
                                           int32_t layout, int32_t chunk_tokens, int32_t budget_num,
                                           int32_t budget_den, double tau, int32_t skip_rule,
                                           int32_t* idx, int32_t max_rows, int32_t* counts,
                                           void* stream);

/*
 * kvfix_repair_rows -- overwrite the chosen rows with exact ones ([BCR] App. B Algorithm 1;
 * [KVCMAS] Eq. 3): for every chunk c of `desc`, layer and KV head, rows
 * idx[c][0 .. counts[c]) of k_io / v_io get the same rows of k_fresh / v_fresh
 * (`fresh_desc`, the shape of desc).  idx holds max_rows entries per chunk; rows out of
 * range are skipped and flagged (KVFIX_EDEVICE in kvfix_check_status).  Either plane may
 * be skipped by passing NULL for both its pointers.
 */
KVFIX_API kvfix_status kvfix_repair_rows(kvfix_bf16* k_io, kvfix_bf16* v_io, kvfix_kv_desc desc,
                                         const kvfix_bf16* k_fresh, const kvfix_bf16* v_fresh,
                                         kvfix_kv_desc fresh_desc, const int32_t* idx,
                                         int32_t max_rows, const int32_t* counts, void* stream);

/*
 * kvfix_master_select -- the master of a round's cache family.  [TD] section 4.2 ("reuse
 * plan output": the reuse pass accumulates a deviation score per request; the master is
 * the request with the lowest total deviation from the shared blocks, which keeps the
 * mirrors' diffs small) and section 4.3 (master-mirror layout).
 *     totals[a] = sum_{r < R} sum_{j < tokens} (d_k[a R + r][j] + d_v[a R + r][j])
 *     *master   = the agent with the smallest total (ties to the lower index)
 * d_k, d_v : device float [agents * R][tokens] as kvfix_score_topk writes them for a
 *            collective round (unit a R + r); either may be NULL.
 * totals   : device double [agents], summed in double in a fixed order (per agent: thread
 *            t of 256 takes every 256th value, then a tree over threads).
 * master   : device int32 [1].
 */
KVFIX_API kvfix_status kvfix_master_select(const float* d_k, const float* d_v, int32_t agents,
                                           int32_t units_per_agent, int32_t tokens, double* totals,
                                           int32_t* master, void* stream);

/*
 * kvfix_diff_encode_split -- block-sparse diffs with one block list per plane.  [TD]
 * section 5 (the K and V planes share one block index list only when they touch the same
 * blocks).  As kvfix_diff_encode, except that entry i is dirty in plane P iff some bf16
 * word of plane P in it differs from the master's, and each plane has its own list:
 *     mask_k / mask_v       : device uint32[ceil(S*L*nblk/32)]
 *     offsets_k / offsets_v : device int64[S*L*nblk + 1]
 *     payload_k / payload_v : device bf16[capacity_P][bt][kv_heads][head_dim] (one plane)
 * h_entries: optional HOST int64[2] (K, V); if given, the call synchronises and returns
 * KVFIX_ENOSPACE, writing no payload, when a plane's total exceeds its capacity.  If NULL,
 * entries beyond a capacity are skipped and flagged.
 */
KVFIX_API kvfix_status kvfix_diff_encode_split(
    const kvfix_bf16* master_k, const kvfix_bf16* master_v, kvfix_kv_desc master,
    const kvfix_bf16* sib_k, const kvfix_bf16* sib_v, kvfix_kv_desc sib, int32_t block_tokens,
    uint32_t* mask_k, uint32_t* mask_v, int64_t* offsets_k, int64_t* offsets_v,
    kvfix_bf16* payload_k, kvfix_bf16* payload_v, int64_t capacity_k, int64_t capacity_v,
    int64_t* h_entries, void* stream);

/*
 * kvfix_diff_gather_split -- restore every sibling from the master and its per-plane
 * diffs (the lists kvfix_diff_encode_split writes): K blocks from (mask_k, offsets_k,
 * payload_k), V blocks from (mask_v, offsets_v, payload_v); entries_* are the payloads'
 * sizes (an offset beyond them is not read and is flagged).  Otherwise as
 * kvfix_diff_gather.
 */
KVFIX_API kvfix_status kvfix_diff_gather_split(
    const kvfix_bf16* master_k, const kvfix_bf16* master_v, kvfix_kv_desc master,
    const uint32_t* mask_k, const uint32_t* mask_v, const int64_t* offsets_k,
    const int64_t* offsets_v, const kvfix_bf16* payload_k, const kvfix_bf16* payload_v,
    int64_t entries_k, int64_t entries_v, int32_t siblings, int32_t block_tokens,
    kvfix_bf16* out_k, kvfix_bf16* out_v, kvfix_kv_desc out, void* stream);

/*
 * kvfix_diff_restore_split -- kvfix_diff_restore from per-plane diffs (the lists
 * kvfix_diff_encode_split writes): the restored K block of a sibling comes from
 * (mask_k, offsets_k, payload_k), its V block from (mask_v, offsets_v, payload_v); a
 * plane whose block is clean is read from the master.  entries_* are the payloads' sizes
 * (an offset beyond them is not read and is flagged).  Re-alignment, slot mapping, pool
 * layout, validation and errors as for kvfix_diff_restore; the output is the same bits
 * as kvfix_diff_restore's on the joint lists of the same siblings.
 */
KVFIX_API kvfix_status kvfix_diff_restore_split(
    const kvfix_bf16* master_k, const kvfix_bf16* master_v, kvfix_kv_desc master,
    const uint32_t* mask_k, const uint32_t* mask_v, const int64_t* offsets_k,
    const int64_t* offsets_v, const kvfix_bf16* payload_k, const kvfix_bf16* payload_v,
    int64_t entries_k, int64_t entries_v, int32_t siblings, int32_t block_tokens,
    const int32_t* delta, double rope_base, const int32_t* slot_mapping, kvfix_bf16* pool_k,
    kvfix_bf16* pool_v, kvfix_kv_desc pool, void* stream);

/*
 * kvfix_anchor_gate_correct -- kvfix_anchor_gate and kvfix_anchor_correct in one pass over
 * the sources: the gate's value-plane distances (prefix k) come from the same
 * reconstructions as the value plane's token weights, the gate is decided on the device,
 * and only accepted segments are corrected (rejected ones keep their outputs; their
 * weights are still written).  Arguments as for the two calls; `accept` is an output here.
 * The gate's squares are summed per thread over the features, folded per warp by a fixed
 * tree and then over the warps in a fixed order, so d differs from kvfix_anchor_gate's in
 * the last bits (and is deterministic).
 * workspace: at least kvfix_anchor_gate_workspace_bytes(src, anchors, src.tokens).
 * head_dim 64 or 128.
 */
KVFIX_API kvfix_status kvfix_anchor_gate_correct(
    const kvfix_bf16* k_src, const kvfix_bf16* v_src, kvfix_kv_desc src, const kvfix_bf16* a_c_k,
    const kvfix_bf16* b_ct_k, const kvfix_bf16* a_c_v, const kvfix_bf16* b_ct_v,
    const kvfix_bf16* a_d_k, const kvfix_bf16* b_dt_k, const kvfix_bf16* a_d_v,
    const kvfix_bf16* b_dt_v, int32_t anchors, int32_t rank, int32_t prefix, double temperature,
    double tau, const int32_t* delta, double rope_base, double* d, double* g, double* hbar,
    int32_t* accept, float* w_k, float* w_v, kvfix_bf16* k_out, kvfix_bf16* v_out,
    kvfix_kv_desc out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvfix_selftest_wait -- exercise the bounded wait that every pipelined kernel uses, with
 * no hang: one warp waits on a barrier phase that never completes and then on the device
 * int32 *flag (optional; 0 = not set), each for at most limit_cycles SM clocks, and records
 * a timeout in the device status word, which kvfix_check_status reports as KVFIX_ETIMEOUT
 * (and clears).  The kernel returns in about 2 * limit_cycles clocks; the context stays
 * usable.  limit_cycles in [1, 4e9].
 */
KVFIX_API kvfix_status kvfix_selftest_wait(int64_t limit_cycles, const int32_t* flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVFIX_H */
