// lowrank_draft.cu -- kvfix_lowrank_draft: the rank-r delta of the key plane and the
// draft-query scoring of the corrected keys in one pass over the cache.
//
// Method: KVCMAS Eq. 4, 7, 8 (the corrected keys are the reference keys plus a delta
// stored as the low-rank product A B); Budgeted Cache Repair section 3 ("The repair":
// the rows are ranked by the softmax attention mass of the draft queries over the
// predicted keys, summed over the layers after the first, the draft steps and the query
// heads) and App. B Algorithm 2 (grouped-query keys expanded to the query heads).
//
// kvfix_lowrank_apply followed by kvfix_draft_rank reads every corrected key twice: once
// to write it and once to score it.  Here the scoring reads the corrected 128-row key
// tile from shared memory, where the low-rank epilogue has just written it for its store.
//
// Persistent and cooperative (every CTA resident at once, one per SM): each group of 8
// consecutive CTAs walks (chunk, layer, KV head) units u = group, group + groups, ...;
// CTA k of a group takes key tiles [k tpc, (k+1) tpc) of every unit.  (Groups are formed
// in software rather than as thread-block clusters: a cluster of 8 one-per-SM CTAs must
// sit in one GPC, which leaves a fifth of the SMs without one.)  Roles:
//   warp 0      TMA producer: the x tile (128 rows x D in 64-column boxes, 128-byte
//               swizzle) and the A tile (128 x r) of each stage of a ring;
//   warp 1      low-rank MMA issuer: per tile A B (M = 128, N = D, K = r) into one of two
//               tensor-memory accumulators;
//   warps 2..5  low-rank epilogue: accumulator + x, rounded to bf16 and written in place
//               (the stage becomes the corrected tile), stored by TMA;
//   warp 11     logits MMA issuer: once a stage holds corrected keys, K~ Q^T (M = 128
//               keys, N = 16 query rows, K = D) into tensor-memory columns [16 i, 16 i + 16):
//               a unit's logits never leave tensor memory;
//   warps 7..10 softmax, after a unit's last logits: max and sum of exp per query row
//               over the CTA's keys; the group's 8 (max, sum) exchanged through a small
//               global-memory area (values, then a per-unit flag with release semantics,
//               read with acquire semantics); then each key's mass
//               sum_q exp(z - max_q) / sum_q to the workspace.  The arithmetic and its
//               order are those of kvfix_draft_rank's cluster kernel, so the masses equal
//               the unfused call's bit for bit.  Running in warps of their own, the
//               softmax of one unit overlaps the low-rank stream of the next;
//   warp 6      each unit's B (r x D) and draft queries (16 x D, zero rows past the
//               group) into two alternating shared-memory buffers, K-major.
// Tensor memory (the whole 512 columns; one CTA per SM): logits in [0, 256), the two
// accumulators in [256, 256 + 2 D).  A unit's first logits wait until the softmax of the
// previous unit has read its logits; the ring's stages are the slack.  Every wait is
// bounded; past the limit a CTA flags a timeout, skips the rest of its work but still
// publishes every exchange, so no CTA of its group is held.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "softmax.cuh"
#include "tc.cuh"

namespace kvfix {

static __device__ unsigned int g_status_ldraft;

unsigned read_status_lowrank_draft(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_ldraft, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_ldraft, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

constexpr int kLdGroup = 8;           // CTAs that share a unit
constexpr int kLdMaxGroups = 64;      // the exchange area is sized for up to 512 CTAs
constexpr int kLdThreads = 384;       // warps: 0 TMA, 1 low-rank MMA, 2..5 epilogue, 6 B/Q loader,
                                      // 7..10 softmax, 11 logits MMA
constexpr int kLdRows = 128;          // rows per tile (MMA M)
constexpr int kLdQ = 16;              // query rows per unit, padded (logits MMA N)
constexpr int kLdMaxStages = 5;
constexpr int kLdSmemLimit = 227 * 1024;
constexpr int kLdLogitCols = 256;     // logits of up to 16 tiles per CTA
constexpr int kLdMaxTiles = kLdLogitCols / 16;
constexpr int kLdMinSmem = 120 * 1024;  // keeps one CTA per SM: it holds all of tensor memory
constexpr float kLdLog2e = 1.4426950408889634f;

template <int D, int RANK>
struct LdCfg {
    static constexpr int kXBytes = kLdRows * D * 2;             // x tile, then the corrected tile
    static constexpr int kABytes = kLdRows * RANK * 2;          // A tile
    static constexpr int kStage = ((kXBytes + kABytes) + 1023) / 1024 * 1024;
    static constexpr int kBBytes = D * RANK * 2;                // one unit's B
    static constexpr int kQBytes = kLdQ * D * 2;                // one unit's draft queries
    static constexpr int kFixed = 1024 /*alignment slack*/ + 2 * kBBytes + 2 * kQBytes;
    static constexpr int kFit = (kLdSmemLimit - kFixed) / kStage;
    static constexpr int kStages = kFit < kLdMaxStages ? kFit : kLdMaxStages;
    static constexpr int kNeed = kFixed + kStages * kStage;
    static constexpr int kSmem = kNeed > kLdMinSmem ? kNeed : kLdMinSmem;
    static constexpr int kASwizzleBytes = RANK * 2;             // 32, 64 or 128
    static constexpr uint32_t kALayout = RANK == 16 ? 6u : RANK == 32 ? 4u : 2u;
};

struct LdArgs {
    const uint16_t* B;   // [C][L][H][RANK][D]
    const uint16_t* q;   // [C][L][steps][Hq][D]
    float* contrib;      // [C][L - layer_begin][H][n]
    float* xval;         // [group][2 parities][8 ranks][16 rows][max, sum]
    int* xflag;          // [group][2 parities][8 ranks]: 1 + index of the last scored unit published
    int C, L, H, n, steps, q_heads, layer_begin, G, tiles, tpc, units;
};

// Bytes of the exchange area that follows the per-key masses in the workspace.
constexpr size_t kLdXchValBytes = sizeof(float) * kLdMaxGroups * 2 * kLdGroup * kLdQ * 2;
constexpr size_t kLdXchFlagBytes = sizeof(int) * kLdMaxGroups * 2 * kLdGroup;
constexpr size_t kLdXchBytes = kLdXchValBytes + kLdXchFlagBytes;

__device__ __forceinline__ int ld_vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <int D, int RANK>
__global__ void __launch_bounds__(kLdThreads, 1)
lowrank_draft_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_out,
                     const __grid_constant__ CUtensorMap tm_a, LdArgs args) {
    using K = LdCfg<D, RANK>;
    constexpr int S = K::kStages;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[S], empty[S], kready[S], accf[2], acce[2], bqf[2], bqe[2],
        lfull[kLdMaxTiles], lfree, drain_lr, drain_qk;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float red_m[4][kLdQ], red_s[4][kLdQ];
    __shared__ float fin_m[kLdQ], fin_inv[kLdQ];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* bsm0 = smem + S * K::kStage;   // two B buffers, K-major canonical, no swizzle
    unsigned char* qsm0 = bsm0 + 2 * K::kBBytes;  // two query buffers, likewise
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = blockIdx.x % kLdGroup;
    const int cid = blockIdx.x / kLdGroup, ncl = gridDim.x / kLdGroup;
    const int n = args.n, H = args.H, L = args.L;
    const int tile0 = rank * args.tpc;
    const int ntiles = max(0, min(args.tpc, args.tiles - tile0));
    auto unit_of = [&](int u, int& c, int& l, int& h) {
        h = u % H;
        l = (u / H) % L;
        c = u / (H * L);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);   // the logits MMA (or its stand-in) and the store
            mbar_init(&kready[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accf[a], 1);
            mbar_init(&acce[a], 4);
            mbar_init(&bqf[a], 1);
            mbar_init(&bqe[a], 2);     // both MMA issuers are done with the buffer
        }
        for (int i = 0; i < kLdMaxTiles; ++i) mbar_init(&lfull[i], 1);  // tile i's logits are in
        mbar_init(&lfree, 1);
        mbar_init(&drain_lr, 1);
        mbar_init(&drain_qk, 1);
        fence_mbar_init();
        abort_flag = 0;
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_out);
        prefetch_tensormap(&tm_a);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t tacc = tmem + kLdLogitCols;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int u = cid; ok && u < args.units && !ld_vload(&abort_flag); u += ncl) {
                int c, l, h;
                unit_of(u, c, l, h);
                const long long arow = (((long long)c * L + l) * H + h) * n;
                for (int i = 0; i < ntiles; ++i, ++g) {
                    const int s = g % S;
                    if (g >= S && !mbar_wait(&empty[s], (unsigned)(g / S - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    unsigned char* st = smem + s * K::kStage;
                    const int t0 = (tile0 + i) * kLdRows;
                    mbar_arrive_expect_tx(&full[s], (unsigned)(K::kXBytes + K::kABytes));
                    for (int hb = 0; hb < D / 64; ++hb)
                        tma_load_4d(st + hb * (kLdRows * 128), &tm_x, h * D + 64 * hb, t0, l, c, &full[s]);
                    tma_load_2d(st + K::kXBytes, &tm_a, 0, (int)(arow + t0), &full[s]);
                }
            }
            if (!ok) atomicOr(&abort_flag, 1);
            if (ld_vload(&abort_flag))  // copies still in flight land before the CTA leaves (bounded)
                for (int k = max(0, g - S); k < g; ++k) mbar_wait(&full[k % S], (unsigned)(k / S) & 1u);
        }
    } else if (warp == 6) {
        // ------------------------------------------------------------ B and query loader
        const int group = args.q_heads / H;
        int j = 0;
        for (int u = cid; u < args.units; u += ncl, ++j) {
            if (ld_vload(&abort_flag)) break;
            int c, l, h;
            unit_of(u, c, l, h);
            const int buf = j & 1;
            if (j >= 2) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&bqe[buf], (unsigned)(j / 2 - 1) & 1u);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) atomicOr(&abort_flag, 1);
                    break;
                }
            }
            // 16-byte pieces, all of a batch loaded before any is stored.  B piece p = row k,
            // elements [e0, e0 + 8): element (k, e) sits at (e%8)*16 + (e/8)*(RANK/8)*128 +
            // (k/8)*128 + (k%8)*2 (K-major, no swizzle).
            unsigned char* bsm = bsm0 + buf * K::kBBytes;
            const uint4* Bu = reinterpret_cast<const uint4*>(args.B + (((long long)c * L + l) * H + h) * RANK * D);
            constexpr int kBPieces = RANK * D / 8;
            for (int p0 = 0; p0 < kBPieces; p0 += 32 * 8) {
                uint4 v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int p = p0 + 32 * q + lane;
                    if (p < kBPieces) v[q] = __ldg(Bu + p);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int p = p0 + 32 * q + lane;
                    if (p >= kBPieces) continue;
                    const int k = p / (D / 8), e8 = p % (D / 8);
                    unsigned char* dst = bsm + e8 * (RANK / 8) * 128 + (k / 8) * 128 + (k % 8) * 2;
                    const uint16_t* hv = reinterpret_cast<const uint16_t*>(&v[q]);
#pragma unroll
                    for (int t = 0; t < 8; ++t) *reinterpret_cast<uint16_t*>(dst + t * 16) = hv[t];
                }
            }
            if (l >= args.layer_begin) {
                // query row i = t*group + m <-> q[c][l][t][h*group + m], zero past the group;
                // piece (i, e8) = elements [8 e8, 8 e8 + 8) at (i%8)*16 + (i/8)*(D/8)*128 + e8*128
                unsigned char* qsm = qsm0 + buf * K::kQBytes;
                constexpr int kQPieces = kLdQ * D / 8;
                uint4 v[kQPieces / 32];
#pragma unroll
                for (int q = 0; q < kQPieces / 32; ++q) {
                    const int p = 32 * q + lane, i = p / (D / 8), e8 = p % (D / 8);
                    v[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (i < args.G) {
                        const int t = i / group, m = i % group;
                        v[q] = __ldg(reinterpret_cast<const uint4*>(
                            args.q + ((((long long)c * L + l) * args.steps + t) * args.q_heads + h * group + m) * D) + e8);
                    }
                }
#pragma unroll
                for (int q = 0; q < kQPieces / 32; ++q) {
                    const int p = 32 * q + lane, i = p / (D / 8), e8 = p % (D / 8);
                    *reinterpret_cast<uint4*>(qsm + (i % 8) * 16 + (i / 8) * (D / 8) * 128 + e8 * 128) = v[q];
                }
            }
            fence_proxy_async_smem();  // generic writes -> read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&bqf[buf]);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ low-rank MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc_bf16(kLdRows, D);
            int g = 0, j = 0;
            bool ok = true;
            for (int u = cid; ok && u < args.units; u += ncl, ++j) {
                const int buf = j & 1;
                if (ld_vload(&abort_flag) || !mbar_wait(&bqf[buf], (unsigned)(j / 2) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned char* bsm = bsm0 + buf * K::kBBytes;
                for (int i = 0; i < ntiles; ++i, ++g) {
                    const int s = g % S, a = g & 1;
                    if (!mbar_wait(&full[s], (unsigned)(g / S) & 1u) ||
                        (g >= 2 && !mbar_wait(&acce[a], (unsigned)(g / 2 - 1) & 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const unsigned char* at = smem + s * K::kStage + K::kXBytes;
#pragma unroll
                    for (int kk = 0; kk < RANK / 16; ++kk) {
                        const uint64_t adesc = tc_smem_desc(at + 32 * kk, 16, 8 * K::kASwizzleBytes, K::kALayout);
                        const uint64_t bdesc = tc_smem_desc(bsm + 256 * kk, 128, (RANK / 8) * 128, 0);
                        tc_mma_bf16(tacc + a * D, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&accf[a]);
                }
                if (ok) tc_commit(&bqe[buf]);  // this unit's B is no longer read
            }
            if (!ok) atomicOr(&abort_flag, 1);
            tc_commit(&drain_lr);  // every MMA this thread issued has completed (bounded wait)
            mbar_wait(&drain_lr, 0u);
        }
    } else if (warp == 11) {
        // ------------------------------------------------------------ logits MMA issuer
        // the logits of a tile once the epilogue has turned its stage into corrected keys
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc_bf16(kLdRows, kLdQ);
            int g = 0, j = 0, sidx_next = 0;
            bool ok = true;
            for (int u = cid; ok && u < args.units; u += ncl, ++j) {
                int c, l, h;
                unit_of(u, c, l, h);
                const int buf = j & 1;
                const bool scored = l >= args.layer_begin;
                const int sidx = scored ? sidx_next++ : 0;
                if (ld_vload(&abort_flag) || !mbar_wait(&bqf[buf], (unsigned)(j / 2) & 1u)) {
                    ok = false;
                    break;
                }
                // A scored unit starts once the softmax of the previous one has read its logits:
                // its logits overwrite those columns, and its completion signal (one phase of
                // a one-arrival barrier) must not run ahead of the softmax that waits for it,
                // also when this CTA has no tiles.
                if (scored && sidx > 0 && !mbar_wait(&lfree, (unsigned)(sidx - 1) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned char* qsm = qsm0 + buf * K::kQBytes;
                for (int i = 0; i < ntiles; ++i, ++g) {
                    const int s = g % S;
                    if (!mbar_wait(&kready[s], (unsigned)(g / S) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!scored) {
                        mbar_arrive(&empty[s]);  // the low-rank MMA finished before the epilogue ran
                        continue;
                    }
                    const unsigned char* kt = smem + s * K::kStage;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t adesc = tc_smem_desc(kt + (kk / 4) * (kLdRows * 128) + 32 * (kk % 4), 16, 1024, 2);
                        const uint64_t bdesc = tc_smem_desc(qsm + 256 * kk, 128, (D / 8) * 128, 0);
                        tc_mma_bf16(tmem + kLdQ * i, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                    tc_commit(&lfull[i]);  // the softmax may read this tile's logits
                }
                if (!ok) break;
                tc_commit(&bqe[buf]);  // this unit's queries are no longer read
            }
            if (!ok) atomicOr(&abort_flag, 1);
            tc_commit(&drain_qk);
            mbar_wait(&drain_qk, 0u);
        }
    } else if (warp >= 2 && warp <= 5) {
        // ------------------------------------------------------------ low-rank epilogue
        const int wq = warp & 3;
        const int m = 32 * wq + lane;           // tile row = tensor-memory lane of this thread
        const int et = threadIdx.x - 64;        // 0..127
        int g = 0, prev_store = -1;             // prev_store: thread et == 0 only
        for (int u = cid; u < args.units; u += ncl) {
            int c, l, h;
            unit_of(u, c, l, h);
            for (int i = 0; i < ntiles; ++i, ++g) {
                const int s = g % S, a = g & 1;
                bool live = !ld_vload(&abort_flag);
                if (live && !mbar_wait(&accf[a], (unsigned)(g / 2) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    live = false;
                }
                live = __all_sync(0xffffffffu, live);  // tensor-memory loads are warp-wide
                tc_fence_after();
                unsigned char* st = smem + s * K::kStage;
                if (live) {
#pragma unroll
                    for (int jj = 0; jj < D / 32; ++jj) {
                        uint32_t v[32];
                        tmem_ld32(tacc + ((uint32_t)(32 * wq) << 16) + a * D + 32 * jj, v);
                        tmem_wait_ld();
                        unsigned char* hb = st + (jj / 2) * (kLdRows * 128) + m * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int chunk = ((32 * jj) % 64) / 8 + q;
                            uint4* p = reinterpret_cast<uint4*>(hb + ((chunk ^ (m & 7)) << 4));
                            float xf[8];
                            unpack8(*p, xf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) xf[e] += __uint_as_float(v[8 * q + e]);
                            *p = pack8(xf);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce[a]);
                fence_proxy_async_smem();  // the corrected tile -> TMA store and logits MMA
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (et == 0) {
                    if (live) {
                        const int t0 = (tile0 + i) * kLdRows;
                        for (int hb = 0; hb < D / 64; ++hb)
                            tma_store_4d(&tm_out, st + hb * (kLdRows * 128), h * D + 64 * hb, t0, l, c);
                    }
                    bulk_commit();
                    mbar_arrive(&kready[s]);
                    bulk_wait_read<1>();  // the previous tile's store has read its stage
                    if (prev_store >= 0) mbar_arrive(&empty[prev_store]);
                    prev_store = s;
                }
            }
        }
        if (et == 0) {
            bulk_wait_read<0>();
            if (prev_store >= 0) mbar_arrive(&empty[prev_store]);
            bulk_wait<0>();
        }
    } else if (warp >= 7 && warp <= 10) {
        // ------------------------------------------------------------ softmax
        // Warp w reads tensor-memory lanes 32 (w % 4) ...; its partials take slot
        // (w % 4 + 2) % 4, the slot the same lanes have in kvfix_draft_rank's cluster
        // kernel, so the partials are added in the same order.
        const int wq = warp & 3, ew = (wq + 2) & 3;
        const int et = threadIdx.x - 224;       // 0..127
        const int key_in_tile = 32 * wq + lane;
        const float scale = rsqrtf((float)D) * kLdLog2e;  // logits in base-2 units
        const int nl = L - args.layer_begin;
        int sidx = 0;
        for (int u = cid; u < args.units; u += ncl) {
            int c, l, h;
            unit_of(u, c, l, h);
            if (l < args.layer_begin) continue;
            // one pass over the unit's logits as they land, tile by tile: per query row the
            // running maximum and rescaled sum (softmax.cuh), as in kvfix_draft_rank
            bool live = !ld_vload(&abort_flag);
            float mx[kLdQ], sm[kLdQ];
#pragma unroll
            for (int q = 0; q < kLdQ; ++q) {
                mx[q] = -INFINITY;
                sm[q] = 0.f;
            }
            for (int i = 0; i < ntiles; ++i) {
                if (live && !mbar_wait(&lfull[i], (unsigned)sidx & 1u)) {
                    atomicOr(&abort_flag, 1);
                    live = false;
                }
                live = __all_sync(0xffffffffu, live);
                if (!live) break;
                tc_fence_after();
                const int key = (tile0 + i) * kLdRows + key_in_tile;
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * wq) << 16) + kLdQ * i, v);
                tmem_wait_ld();
                if (key < n) {
#pragma unroll
                    for (int q = 0; q < kLdQ; ++q) online_add(mx[q], sm[q], __uint_as_float(v[q]) * scale);
                }
            }
#pragma unroll
            for (int q = 0; q < kLdQ; ++q) warp_combine(mx[q], sm[q]);
            if (lane == 0)
#pragma unroll
                for (int q = 0; q < kLdQ; ++q) {
                    red_m[ew][q] = mx[q];
                    red_s[ew][q] = sm[q];
                }
            asm volatile("bar.sync 2, 128;" ::: "memory");
            const int xb = sidx & 1;
            float* xv = args.xval + (((long long)cid * 2 + xb) * kLdGroup) * kLdQ * 2;  // [8 ranks][16][2]
            int* xf = args.xflag + ((long long)cid * 2 + xb) * kLdGroup;             // [8 ranks]
            if (et < kLdQ) {  // publish this CTA's (max, sum) of query row et
                const float m4[4] = {red_m[0][et], red_m[1][et], red_m[2][et], red_m[3][et]};
                const float s4[4] = {red_s[0][et], red_s[1][et], red_s[2][et], red_s[3][et]};
                float cm, cs;
                combine4(m4, s4, cm, cs);
                xv[(rank * kLdQ + et) * 2] = cm;
                xv[(rank * kLdQ + et) * 2 + 1] = cs;
                __threadfence();
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (et == 0) st_release_gpu(xf + rank, sidx + 1);
            if (et < kLdQ) {  // every row's thread waits for the 8 flags, then combines in rank order
                bool got = !ld_vload(&abort_flag);
                const long long t0 = clock64();
                for (int k = 0; got && k < kLdGroup; ++k)
                    while (ld_acquire_gpu(xf + k) != sidx + 1)
                        if (clock64() - t0 > kWaitCycles) {
                            atomicOr(&abort_flag, 1);
                            got = false;
                            break;
                        }
                float mg = -INFINITY;
                for (int k = 0; k < kLdGroup; ++k) mg = fmaxf(mg, __ldcg(xv + (k * kLdQ + et) * 2));
                float ssum = 0.f;
                for (int k = 0; k < kLdGroup; ++k) {
                    const float mk = __ldcg(xv + (k * kLdQ + et) * 2);
                    if (mk != -INFINITY) ssum += __ldcg(xv + (k * kLdQ + et) * 2 + 1) * exp2f(mk - mg);
                }
                fin_m[et] = mg;
                fin_inv[et] = ssum > 0.f ? 1.0f / ssum : 0.f;
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");
            live = __all_sync(0xffffffffu, live && !ld_vload(&abort_flag));
            float* out = args.contrib + (((long long)c * nl + (l - args.layer_begin)) * H + h) * n;
            for (int i = 0; i < ntiles && live; ++i) {
                const int key = (tile0 + i) * kLdRows + key_in_tile;
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * wq) << 16) + kLdQ * i, v);
                tmem_wait_ld();
                float acc = 0.f;
                for (int q = 0; q < args.G; ++q) acc += exp2f(__uint_as_float(v[q]) * scale - fin_m[q]) * fin_inv[q];
                if (key < n) out[key] = acc;
            }
            tc_fence_before();
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (et == 0) mbar_arrive(&lfree);  // the logits columns may be overwritten
            ++sidx;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(&g_status_ldraft, FLAG_TIMEOUT);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// 4-D map of a plane with (64-element x 128-row) boxes and 128-byte swizzle.
static cudaError_t encode_rows64(CUtensorMap* map, const void* base, const Plane& p) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[4], strides[3];
    plane_map_strides(p, dims, strides);
    cuuint32_t box[4] = {64, (cuuint32_t)kLdRows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int RANK>
static cudaError_t launch_ld_t(const uint16_t* x, const Plane& p, const uint16_t* A, const uint16_t* B,
                               uint16_t* out, const Plane& op, LdArgs args, cudaStream_t s) {
    using K = LdCfg<D, RANK>;
    CUtensorMap tx, to, ta;
    cudaError_t e;
    if ((e = encode_rows64(&tx, x, p)) != cudaSuccess) return e;
    if ((e = encode_rows64(&to, out, op)) != cudaSuccess) return e;
    auto enc = tensor_map_encoder();
    const long long rows = (long long)p.chunks * p.layers * p.heads * p.tokens;
    cuuint64_t adims[2] = {(cuuint64_t)RANK, (cuuint64_t)rows};
    cuuint64_t astr[1] = {(cuuint64_t)RANK * 2};
    cuuint32_t abox[2] = {(cuuint32_t)RANK, (cuuint32_t)kLdRows};
    cuuint32_t aestr[2] = {1, 1};
    if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A), adims, astr, abox, aestr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(K::kASwizzleBytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    args.B = B;
    auto kernel = lowrank_draft_kernel<D, RANK>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K::kSmem);
    if (e != cudaSuccess) return e;
    // Persistent and cooperative: one CTA per SM (each holds all of its SM's tensor
    // memory), in groups of 8, at most one group per unit.  The cooperative launch
    // guarantees that every CTA of a group is resident while its peers wait for it.
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kLdThreads, K::kSmem)) != cudaSuccess)
        return e;
    const long long groups = std::min<long long>(std::min(sms * std::min(per_sm, 1) / kLdGroup, kLdMaxGroups),
                                                 args.units);
    if (groups < 1) return cudaErrorInvalidConfiguration;
    if ((e = cudaMemsetAsync(args.xflag, 0, kLdXchFlagBytes, s)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(groups * kLdGroup));
    cfg.blockDim = dim3(kLdThreads);
    cfg.dynamicSmemBytes = K::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tx, to, ta, args);
}

size_t lowrank_draft_workspace_bytes(const kvfix_kv_desc& d, int layer_begin) {
    return draft_workspace_bytes(d, layer_begin) + kLdXchBytes;
}

cudaError_t launch_lowrank_draft(const uint16_t* x, const kvfix_kv_desc& d, const uint16_t* A, const uint16_t* B,
                                 int rank, uint16_t* out, const kvfix_kv_desc& od, const uint16_t* q, int steps,
                                 int q_heads, int layer_begin, int k_rows, int32_t* idx, double* scores, void* ws,
                                 cudaStream_t s) {
    Plane p = plane_of(d), op = plane_of(od);
    if (p.chunks == 0 || p.layers == 0 || p.tokens == 0) return cudaSuccess;
    LdArgs a;
    a.q = q;
    a.contrib = static_cast<float*>(ws);
    // the exchange area follows the per-key masses (whose size is a multiple of 256 bytes)
    unsigned char* xch = static_cast<unsigned char*>(ws) + draft_workspace_bytes(d, layer_begin);
    a.xval = reinterpret_cast<float*>(xch);
    a.xflag = reinterpret_cast<int*>(xch + kLdXchValBytes);
    a.C = p.chunks;
    a.L = p.layers;
    a.H = p.heads;
    a.n = p.tokens;
    a.steps = steps;
    a.q_heads = q_heads;
    a.layer_begin = layer_begin;
    a.G = steps * (q_heads / p.heads);
    a.tiles = (p.tokens + kLdRows - 1) / kLdRows;
    a.tpc = (a.tiles + kLdGroup - 1) / kLdGroup;
    a.units = p.chunks * p.layers * p.heads;
    if (kLdQ * a.tpc > kLdLogitCols) return cudaErrorInvalidValue;  // tokens <= 16384
    cudaError_t e;
    if (p.dim == 128) {
        e = rank == 16 ? launch_ld_t<128, 16>(x, p, A, B, out, op, a, s)
          : rank == 32 ? launch_ld_t<128, 32>(x, p, A, B, out, op, a, s)
                       : launch_ld_t<128, 64>(x, p, A, B, out, op, a, s);
    } else {
        e = rank == 16 ? launch_ld_t<64, 16>(x, p, A, B, out, op, a, s)
          : rank == 32 ? launch_ld_t<64, 32>(x, p, A, B, out, op, a, s)
                       : launch_ld_t<64, 64>(x, p, A, B, out, op, a, s);
    }
    if (e != cudaSuccess) return e;
    const long long units_per_chunk = (long long)(p.layers > layer_begin ? p.layers - layer_begin : 0) * p.heads;
    return launch_draft_finish(a.contrib, p.chunks, p.tokens, units_per_chunk, k_rows, idx, scores, s);
}

}  // namespace kvfix
