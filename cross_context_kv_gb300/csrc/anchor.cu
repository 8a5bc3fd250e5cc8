// anchor.cu -- anchor-pool correction of a reused segment (kvfix_anchor_gate,
// kvfix_anchor_correct).
//
// Method: KVCMAS section 3.3 (anchors keep their base cache and delta corrections as
// low-rank factors, Eq. 7; the transition correction is the weighted sum of the anchors'
// deltas, Eq. 8, applied to the aligned source cache, Eq. 4) and App. A.3 (reliability
// gate on the value states over a prefix, Eq. 9-11; token-wise interpolation weights
// from the mean absolute source-to-anchor distance, keys and values separately, softmax
// with T = 1; keys matched in canonical positions and then aligned to their targets).
//
// Factor layout (one plane): A [segment][anchor][layer][token][r], and the second factor
// stored transposed, Bt [segment][anchor][layer][feature][r] (feature = head*D + dim),
// so that both MMA operands are K-major with K = r.
//
// Blackwell path, three kernels; the two big ones are persistent (one CTA per SM slot
// walks the (128-row tile, layer, plane and segment) units, its rings running on from
// one unit to the next):
//   anchor_dist_kernel   per unit: the anchors' base
//                        rows A_v B_v are built 128 features at a time by tcgen05.mma
//                        (M = 128 rows, N = 128, K = r) into four tensor-memory buffers,
//                        while eight epilogue warps fold |x - rec| (token weights) or
//                        (x - rec)^2 (gate) into per-row, per-anchor sums; x chunks and Bt
//                        stream through TMA rings fed by two producer lanes.
//   anchor_gate_kernel   per segment: the gate's distances, softmax, normalised entropy.
//   anchor_apply_kernel  per unit: the anchors' delta factors
//                        are scaled by the token weights in shared memory and multiplied by
//                        the stacked Bt (K = V*r) head by head into tensor memory; the
//                        epilogue adds the aligned source (keys rotated) and stores by TMA.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc.cuh"

namespace kvfix {

static __device__ unsigned int g_status_anchor;

unsigned read_status_anchor(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_anchor, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_anchor, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

__device__ __forceinline__ int anchor_vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// Named barrier over the epilogue warps that also ORs a predicate across them, so that a
// failed wait in any of them stops all of them at the same step.
template <int ID, int N>
__device__ __forceinline__ bool bar_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " barrier.cta.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(ID), "n"(N)
        : "memory");
    return r != 0;
}

constexpr int kAnRows = 128;          // rows per tile (MMA M)
constexpr int kAnMaxAnchors = 16;
constexpr int kAnSmemLimit = 227 * 1024;

// ------------------------------------------------------------------ distances

constexpr int kAdThreads = 352;       // warp 0 TMA, warps 1 and 10 MMA, warps 2..9 epilogue
constexpr int kAdCols = 128;          // features per chunk (MMA N)
constexpr int kAdSlots = 4;           // tensor-memory accumulators of 128 columns
constexpr int kAdMaxB = 16;           // Bt ring entries (one anchor's chunk each)
constexpr int kAdMaxX = 4;            // x chunk buffers
constexpr int kAdXBytes = kAnRows * kAdCols * 2;  // x chunk: two 64-feature boxes, 128-byte swizzle
constexpr int kAdEpi = 256;           // epilogue threads

enum { kAdWeights = 0, kAdGate = 1, kAdBoth = 2 };

struct AdArgs {
    int V, L, n, F, C;
    int rows;            // rows of the tile range: n (weights) or the gate prefix k
    int tiles;           // ceil(rows / 128)
    int nb, nx;          // Bt ring entries, x chunk buffers
    float inv_T;
    float* w[2];         // weights mode: [C][L][n][V] per plane
    float* partial;      // gate mode, and both mode's value plane: [C][L][tiles][V]
    int gate_rows;       // both mode: the gate's prefix k
    const int32_t* accept;  // weights mode: [C] or null; rejected segments are skipped
};

template <int R>
struct AdCfg {
    static constexpr int kRowBytes = R * 2;                       // 32, 64 or 128
    static constexpr uint32_t kLayout = R == 16 ? 6u : R == 32 ? 4u : 2u;
    static constexpr int kABytes = kAnRows * kRowBytes;           // one anchor's A tile
    static constexpr int kBBytes = kAdCols * kRowBytes;           // one anchor's Bt chunk
};

// Persistent: CTA i takes the units (128-row tile, layer, plane and segment) i, i + grid,
// ...; the x, Bt and tensor-memory rings run on from one unit to the next, and a unit's A
// tiles are loaded once the previous unit's MMAs have committed ("adone"), so the next
// unit's loads overlap the previous one's epilogue.  Per unit, for each 128-feature chunk
// the x tile is staged once; each thread takes its row's 64 of the chunk's features into
// registers as -x and writes them into the tensor-memory slot of each (chunk, anchor) step
// before the step's MMA (M = 128 rows, N = 128 features, K = r) accumulates the anchor's
// reconstruction onto them, so the epilogue reads rec - x from four rotating slots.
// MODE kAdWeights: both planes (z = plane * C + c), every row; writes the softmax of
// -mean|x - rec_v| / T per row.  MODE kAdGate: the value plane, rows < k; writes per-tile
// sums of (x - rec_v)^2.  MODE kAdBoth: the weights of both planes and, on the value
// plane, the gate's per-tile sums from the same reconstructions (per-thread sums folded
// per warp and then over the warps in a fixed order).
//
// After an abort a producer waits (bounded) for the copies it armed last on each barrier
// of a ring, so that no bulk copy is still writing shared memory when the CTA leaves;
// item i of a ring of n one-arrival barriers is phase i / n of barrier i % n.
__device__ __forceinline__ void drain_ring(uint64_t* ring, int n, int armed) {
    for (int i = armed > n ? armed - n : 0; i < armed; ++i) mbar_wait(&ring[i % n], (unsigned)(i / n) & 1u);
}

template <int R, int MODE>
__global__ void __launch_bounds__(kAdThreads, 1)
anchor_dist_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_x1,
                   const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_b1,
                   AdArgs args) {
    using K = AdCfg<R>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t xfull[kAdMaxX], xempty[kAdMaxX], bfull[kAdMaxB], bempty[kAdMaxB], tfull[kAdSlots],
        tinit[kAdSlots], afull, adone, mdrain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float gsum[4][kAnMaxAnchors];
    __shared__ float gsq[8][kAnMaxAnchors];  // both mode: per epilogue warp, per anchor
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int V = args.V, NB = args.nb, NX = args.nx;
    unsigned char* asm_ = smem;                             // V A tiles
    unsigned char* xs = smem + V * K::kABytes;              // NX x chunks
    unsigned char* bs = xs + NX * kAdXBytes;                // Bt ring
    float* accs = reinterpret_cast<float*>(bs + NB * K::kBBytes);  // [V][kAdEpi] row sums
    float* gacc = accs + V * kAdEpi;  // both mode: [V][kAdEpi] row sums of squares (gate)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = args.F / kAdCols;
    const int total = chunks * V;                           // (chunk, anchor) steps of a tile
    const int zdim = MODE == kAdGate ? args.C : 2 * args.C;
    const int units = args.tiles * args.L * zdim;           // (tile, layer, plane and segment) units
    // a unit is skipped (by every role alike) when its segment was rejected
    auto unit_of = [&](int w, int& tile, int& l, int& plane, int& c) {
        tile = w % args.tiles;
        const int rest = w / args.tiles;
        l = rest % args.L;
        const int z = rest / args.L;
        plane = MODE == kAdGate ? 0 : z / args.C;
        c = z % args.C;
        return !(MODE != kAdGate && args.accept && args.accept[c] == 0);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NX; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xempty[i], 8);   // the eight epilogue warps
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], 1);
        }
        for (int a = 0; a < kAdSlots; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tinit[a], 8);   // the eight epilogue warps: slot holds -x, ready for the MMA
        }
        mbar_init(&afull, 1);
        mbar_init(&adone, 2);    // both MMA issuers
        mbar_init(&mdrain, 2);
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, kAdSlots * kAdCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 streams A and the x chunks, lane 1 the Bt ring (independent waits); the
        // rings run on across the units of this CTA
        if (lane == 0) {
            prefetch_tensormap(&tm_x0);
            prefetch_tensormap(&tm_x1);
            prefetch_tensormap(&tm_a0);
            prefetch_tensormap(&tm_a1);
            prefetch_tensormap(&tm_b0);
            prefetch_tensormap(&tm_b1);
            int it = 0, an = 0, xn = 0;  // units and x chunks armed
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* mx = plane ? &tm_x1 : &tm_x0;
                const CUtensorMap* ma = plane ? &tm_a1 : &tm_a0;
                const int t0 = tile * kAnRows;
                // the previous unit's MMAs have read their A tiles
                if (it > 0 && !mbar_wait(&adone, (unsigned)(it - 1) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                mbar_arrive_expect_tx(&afull, (unsigned)(V * K::kABytes));
                for (int v = 0; v < V; ++v)
                    tma_load_2d(asm_ + v * K::kABytes, ma, 0, ((c * V + v) * args.L + l) * args.n + t0, &afull);
                ++an;
                bool ok = true;
                for (int j = 0; j < chunks; ++j) {
                    const int jg = it * chunks + j, xi = jg % NX;
                    if (jg >= NX && !mbar_wait(&xempty[xi], (unsigned)(jg / NX - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&xfull[xi], (unsigned)kAdXBytes);
                    for (int b = 0; b < 2; ++b)
                        tma_load_4d(xs + xi * kAdXBytes + b * (kAnRows * 128), mx, j * kAdCols + 64 * b, t0, l, c,
                                    &xfull[xi]);
                    ++xn;
                }
                if (!ok) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                ++it;
            }
            if (anchor_vload(&abort_flag)) {
                drain_ring(&afull, 1, an);
                drain_ring(xfull, NX, xn);
            }
        } else if (lane == 1) {
            int bn = 0, e = 0;  // Bt tiles armed; ring slot of the next
            unsigned ph = 0;     // phase parity of that slot's next fill
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* mb = plane ? &tm_b1 : &tm_b0;
                bool ok = true;
                int j = 0, v = 0;
                for (int q = 0; q < total && !anchor_vload(&abort_flag); ++q) {
                    if (bn >= NB && !mbar_wait(&bempty[e], ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bfull[e], (unsigned)K::kBBytes);
                    tma_load_2d(bs + e * K::kBBytes, mb, 0, ((c * V + v) * args.L + l) * args.F + j * kAdCols, &bfull[e]);
                    ++bn;
                    if (++e == NB) e = 0, ph ^= 1u;
                    if (++v == V) v = 0, ++j;
                }
                if (!ok) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
            }
            if (anchor_vload(&abort_flag)) drain_ring(bfull, NB, bn);
        }
    } else if (warp == 1 || warp == kAdThreads / 32 - 1) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads in two warps issue alternate steps (even and odd step numbers: slots
        // 0, 2 and 1, 3); each commits its own steps.  Ring slots and parities are derived
        // once per unit and then advance without division.
        if (lane == 0) {
            const int par = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = tc_idesc_bf16(kAnRows, kAdCols);
            const uint64_t a_first = tc_smem_desc(asm_, 16, 8 * K::kRowBytes, K::kLayout);
            const uint64_t b_first = tc_smem_desc(bs, 16, 8 * K::kRowBytes, K::kLayout);
            int it = 0;
            bool ok = true;
            for (int w = blockIdx.x; ok && w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                if (!mbar_wait(&afull, (unsigned)it & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int qb = it * total, q0 = (par ^ qb) & 1;
                int qg = qb + q0, e = qg % NB, v = q0 % V;
                unsigned bph = (unsigned)(qg / NB) & 1u;
                for (int q = q0; q < total && !anchor_vload(&abort_flag); q += 2, qg += 2) {
                    const int a = qg & (kAdSlots - 1);
                    if (!mbar_wait(&tinit[a], (unsigned)(qg / kAdSlots) & 1u) || !mbar_wait(&bfull[e], bph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors advance by 16-byte units (shared addresses stay below 256 KB)
                    const uint64_t ad = a_first + (uint64_t)(v * (K::kABytes >> 4));
                    const uint64_t bd = b_first + (uint64_t)(e * (K::kBBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < R / 16; ++kk)
                        tc_mma_bf16(tmem + a * kAdCols, ad + 2 * kk, bd + 2 * kk, idesc, 1u);  // onto -x
                    tc_commit(&bempty[e]);
                    tc_commit(&tfull[a]);
                    e += 2;
                    if (e >= NB) e -= NB, bph ^= 1u;
                    v += 2;
                    while (v >= V) v -= V;
                }
                tc_commit(&adone);  // this issuer's MMAs of the unit are done with the A tiles
                ++it;
            }
            if (!ok) atomicOr(&abort_flag, 1);
            // every MMA issued has completed before the tensor memory is released
            tc_commit(&mdrain);
            mbar_wait(&mdrain, 0u);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Thread et owns row m's 64 features of the chunk.  Before each step's MMA the warps
        // write -x into the step's accumulator slot (tcgen05.st), so that the tensor core
        // leaves rec - x there; the epilogue then folds |rec - x| (and its square for the
        // gate) and accumulates its per-anchor sums in shared memory (accs[v][et]; the
        // anchor loop stays rolled).  A slot is written again right after its values are
        // loaded when its next step lies in the same chunk, else at the start of the next
        // chunk, once that chunk's x is in registers.
        const int ew = warp - 2;              // 0..7
        const int wq = warp & 3;              // TMEM lane quarter this warp may read
        const int half = ew >> 2;             // which 64 of the chunk's 128 features
        const int m = 32 * wq + lane;         // tile row of this thread
        const int et = threadIdx.x - 64;      // 0..255; row m's other half is et ^ 128
        const uint32_t tcol = tmem + ((uint32_t)(32 * wq) << 16) + 64 * half;
        bool ok = true;
        int it = 0;
        for (int w = blockIdx.x; w < units; w += gridDim.x) {
            int tile, l, plane, c;
            if (!unit_of(w, tile, l, plane, c)) continue;
            // the previous unit's reads of accs, gsum and gsq are done; leave together on abort
            if (bar_any<1, 256>(!ok || anchor_vload(&abort_flag))) break;
            const int t0 = tile * kAnRows;
            const bool row_ok = t0 + m < args.rows;
            const bool gate_too = MODE == kAdBoth && plane == 1;
            const bool gate_row = t0 + m < args.gate_rows;
            for (int v = 0; v < V; ++v) accs[v * kAdEpi + et] = 0.f;
            if (gate_too)
                for (int v = 0; v < V; ++v) gacc[v * kAdEpi + et] = 0.f;
            int qg = it * total;
            for (int j = 0; ok && j < chunks; ++j) {
                const int jg = it * chunks + j, xi = jg % NX;
                if (!__all_sync(0xffffffffu, !anchor_vload(&abort_flag) && mbar_wait(&xfull[xi], (unsigned)(jg / NX) & 1u))) {
                    ok = false;
                    break;
                }
                // -x of this row's 64 features of the chunk, as float bit patterns
                uint32_t nx[64];
                const unsigned char* xrow = xs + xi * kAdXBytes + half * (kAnRows * 128) + m * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 u = *reinterpret_cast<const uint4*>(xrow + ((q ^ (m & 7)) << 4));
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        nx[8 * q + 2 * k] = (wd[k] << 16) ^ 0x80000000u;
                        nx[8 * q + 2 * k + 1] = (wd[k] & 0xffff0000u) ^ 0x80000000u;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xempty[xi]);  // x is in registers now
                // the slots of the chunk's first steps (their previous steps were in earlier chunks)
                for (int v = 0; v < V && v < kAdSlots; ++v) {
                    const uint32_t ts = tcol + ((qg + v) & (kAdSlots - 1)) * kAdCols;
                    tmem_st32(ts, nx);
                    tmem_st32(ts + 32, nx + 32);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tinit[(qg + v) & (kAdSlots - 1)]);
                }
#pragma unroll 1
                for (int v = 0; v < V; ++v, ++qg) {
                    const int a = qg & (kAdSlots - 1);
                    if (!__all_sync(0xffffffffu, mbar_wait(&tfull[a], (unsigned)(qg / kAdSlots) & 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t p[32], r[32];
                    tmem_ld32(tcol + a * kAdCols, p);
                    tmem_ld32(tcol + a * kAdCols + 32, r);
                    tmem_wait_ld32(p);
                    tmem_wait_ld32(r);
                    if (v + kAdSlots < V) {
                        // the slot's next step is in this chunk: write -x again now
                        tmem_st32(tcol + a * kAdCols, nx);
                        tmem_st32(tcol + a * kAdCols + 32, nx + 32);
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tinit[a]);
                    }
                    // d = rec - x for features [0, 32) (p) and [32, 64) (r) of this thread's 64
                    float* acc = accs + v * kAdEpi + et;
                    if (MODE == kAdGate) {
                        float2 q2 = make_float2(0.f, 0.f), q2o = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float2 d = make_float2(__uint_as_float(p[2 * e]), __uint_as_float(p[2 * e + 1]));
                            const float2 f = make_float2(__uint_as_float(p[2 * e + 2]), __uint_as_float(p[2 * e + 3]));
                            q2 = __ffma2_rn(d, d, q2);
                            q2o = __ffma2_rn(f, f, q2o);
                        }
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float2 d = make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                            const float2 f = make_float2(__uint_as_float(r[2 * e + 2]), __uint_as_float(r[2 * e + 3]));
                            q2 = __ffma2_rn(d, d, q2);
                            q2o = __ffma2_rn(f, f, q2o);
                        }
                        *acc += (q2.x + q2.y) + (q2o.x + q2o.y);
                    } else {
                        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; e += 4) {
                            s0 += fabsf(__uint_as_float(p[e])) + fabsf(__uint_as_float(p[e + 1]));
                            s1 += fabsf(__uint_as_float(p[e + 2])) + fabsf(__uint_as_float(p[e + 3]));
                            s2 += fabsf(__uint_as_float(r[e])) + fabsf(__uint_as_float(r[e + 1]));
                            s3 += fabsf(__uint_as_float(r[e + 2])) + fabsf(__uint_as_float(r[e + 3]));
                        }
                        *acc += (s0 + s1) + (s2 + s3);
                        if (gate_too) {
                            float2 q2 = make_float2(0.f, 0.f), q2o = make_float2(0.f, 0.f);
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                q2 = __ffma2_rn(make_float2(__uint_as_float(p[e]), __uint_as_float(p[e + 1])),
                                                make_float2(__uint_as_float(p[e]), __uint_as_float(p[e + 1])), q2);
                                q2o = __ffma2_rn(make_float2(__uint_as_float(p[e + 2]), __uint_as_float(p[e + 3])),
                                                 make_float2(__uint_as_float(p[e + 2]), __uint_as_float(p[e + 3])), q2o);
                                q2 = __ffma2_rn(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                                make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), q2);
                                q2o = __ffma2_rn(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])),
                                                 make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), q2o);
                            }
                            gacc[v * kAdEpi + et] += (q2.x + q2.y) + (q2o.x + q2o.y);
                        }
                    }
                }
            }
            tmem_wait_ld();  // no load left in flight (an abort may leave one)
            if (!ok) atomicOr(&abort_flag, 1);
            // the gate's partial of this warp per anchor: its rows below the gate prefix,
            // lanes folded by a fixed tree
            if (MODE == kAdBoth && gate_too) {
                for (int v = 0; v < V; ++v) {
                    float g = gate_row ? gacc[v * kAdEpi + et] : 0.f;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
                    if (lane == 0) gsq[ew][v] = g;
                }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");  // both halves' sums are in accs
            if (MODE == kAdBoth && gate_too && ew == 0 && lane < V && !anchor_vload(&abort_flag)) {
                float x = 0.f;
                for (int w2 = 0; w2 < 8; ++w2) x += gsq[w2][lane];
                args.partial[(((long long)c * args.L + l) * args.tiles + tile) * V + lane] = x;
            }
            if (half == 0 && !anchor_vload(&abort_flag)) {
                // row m's sum per anchor: the first half's plus the second half's
                float* mine = accs + et;
                const float* other = accs + (et ^ 128);
                if (MODE != kAdGate) {
                    if (row_ok) {
                        const float invF = 1.f / (float)args.F;
                        float mmin = (mine[0] + other[0]) * invF;
                        for (int v = 1; v < V; ++v) mmin = fminf(mmin, (mine[v * kAdEpi] + other[v * kAdEpi]) * invF);
                        float z = 0.f;
                        for (int v = 0; v < V; ++v) {
                            const float ev = expf(-((mine[v * kAdEpi] + other[v * kAdEpi]) * invF - mmin) * args.inv_T);
                            mine[v * kAdEpi] = ev;
                            z += ev;
                        }
                        const float iz = 1.f / z;
                        float* wr = (plane ? args.w[1] : args.w[0]) + (((long long)c * args.L + l) * args.n + t0 + m) * V;
                        for (int v = 0; v < V; ++v) wr[v] = mine[v * kAdEpi] * iz;
                    }
                } else {
                    // per-tile sums over the rows, in a fixed order: lanes, then the four warps
                    for (int v = 0; v < V; ++v) {
                        float x = row_ok ? mine[v * kAdEpi] + other[v * kAdEpi] : 0.f;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                        if (lane == 0) gsum[wq][v] = x;
                    }
                }
            }
            if (MODE == kAdGate) {
                asm volatile("bar.sync 1, 256;" ::: "memory");
                if (ew == 0 && lane < V && !anchor_vload(&abort_flag)) {
                    const float x = ((gsum[0][lane] + gsum[1][lane]) + gsum[2][lane]) + gsum[3][lane];
                    args.partial[(((long long)c * args.L + l) * args.tiles + tile) * V + lane] = x;
                }
            }
            ++it;
        }
    }
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(&g_status_anchor, FLAG_TIMEOUT);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kAdSlots * kAdCols);
}

// ------------------------------------------------------------------ gate

// One CTA per segment, one warp per anchor: d_v = sqrt(sum of the per-tile sums over
// layers and tiles, lane j taking every 32nd in double, lanes folded by a fixed tree);
// then warp 0: g = softmax(-d / T), Hbar = -sum g log2 g / log2 V, accepted iff V >= 2 and
// Hbar <= tau.
__global__ void __launch_bounds__(32 * kAnMaxAnchors)
anchor_gate_kernel(const float* __restrict__ partial, int V, int L, int tiles, double T, double tau, double* d,
                   double* g, double* hbar, int32_t* accept) {
    __shared__ double ds[kAnMaxAnchors];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = L * tiles;
    if (warp < V) {
        double s = 0.0;
        for (int lt = lane; lt < n; lt += 32) s += (double)partial[((long long)c * n + lt) * V + warp];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) {
            ds[warp] = sqrt(s);
            d[(long long)c * V + warp] = ds[warp];
        }
    }
    __syncthreads();
    if (warp != 0) return;
    const int v = lane;
    const double dv = v < V ? ds[v] : 0.0;
    double dmin = v < V ? dv : 1e308;
    for (int o = 16; o > 0; o >>= 1) dmin = fmin(dmin, __shfl_xor_sync(0xffffffffu, dmin, o));
    const double e = v < V ? exp(-(dv - dmin) / T) : 0.0;
    double z = e;
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const double gv = e / z;
    if (v < V) g[(long long)c * V + v] = gv;
    double h = (v < V && gv > 0.0) ? -gv * log2(gv) : 0.0;
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    if (v == 0) {
        const double hb = V >= 2 ? h / log2((double)V) : __longlong_as_double(0x7ff8000000000000ll);
        hbar[c] = hb;
        accept[c] = (V >= 2 && hb <= tau) ? 1 : 0;
    }
}

// ------------------------------------------------------------------ apply

constexpr int kApThreads = 352;       // warp 0 TMA loads, warp 1 MMA, warps 2..9 epilogue, warp 10 TMA stores
constexpr int kApEpi = 256;           // epilogue threads: two per tile row
constexpr int kApMaxB = 16;           // Bt ring entries (one anchor's rows of one head group)
constexpr int kApMaxX = 2;            // x head slabs

struct ApArgs {
    int V, L, n, H, C;
    int nb, nx;                       // Bt ring entries and x slabs in use
    int G;                            // heads per MMA group (G * D accumulator columns)
    const float* w[2];                // [C][L][n][V] per plane
    const int32_t* accept;            // [C] or null
    const int32_t* delta;             // [C]
    uint16_t* out[2];                 // only to skip a missing plane
};

template <int D, int R>
struct ApCfg {
    static constexpr int kRowBytes = R * 2;
    static constexpr uint32_t kLayout = R == 16 ? 6u : R == 32 ? 4u : 2u;
    static constexpr int kABytes = kAnRows * kRowBytes;   // one anchor's A tile
    static constexpr int kXBytes = kAnRows * D * 2;       // one head slab of x (64-feature boxes)
    static constexpr int kPairs = D / 4;                  // rotation pairs per epilogue thread and head
};

// Persistent like the distance kernel: CTA i takes the units (tile, layer, plane and
// segment) i, i + grid, ... (plane 0 keys, rotated; 1 values); the x slabs, Bt ring and
// tensor-memory slots run on across units, and a unit's A tiles load once the previous
// unit's MMAs have committed.  The heads go through the tensor core G at a time: one
// MMA chain of N = G * D columns per group (K = V * r), into one of two accumulator
// slots, so that the epilogue of a group overlaps the MMAs of the next.  Each tile row
// is finished by two epilogue threads, each taking half of a head's rotation pairs; a
// head's slab, corrected in place, is stored by the store warp, which frees the slab for
// the next load as soon as the store has read it.
template <int D, int R>
__global__ void __launch_bounds__(kApThreads, 1)
anchor_apply_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_x1,
                    const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                    const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                    const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_b1,
                    ApArgs args, RopeTheta th) {
    using K = ApCfg<D, R>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t afull, ascaled, adone, mdrain, xfull[kApMaxX], xdone[kApMaxX], xempty[kApMaxX],
        bfull[kApMaxB], bempty[kApMaxB], tfull[2], tempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float2 tab[D / 2];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int V = args.V, H = args.H, NB = args.nb, NX = args.nx, G = args.G;
    const int GD = G * D;                                        // accumulator columns of a group
    const int groups = (H + G - 1) / G;
    const int bslot = GD * K::kRowBytes;                         // one anchor's Bt rows of a group
    unsigned char* asm_ = smem;                                  // V scaled A tiles
    unsigned char* xs = asm_ + V * K::kABytes;                   // NX head slabs of x
    unsigned char* bs = xs + NX * K::kXBytes;                    // Bt ring
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int F = H * D;
    const int tiles = (args.n + kAnRows - 1) / kAnRows;
    const int units = tiles * args.L * 2 * args.C;
    // unit w = ((plane * C + c) * L + l) * tiles + tile; missing planes and rejected segments
    // are skipped by every role alike
    auto unit_of = [&](int w, int& tile, int& l, int& plane, int& c) {
        tile = w % tiles;
        const int rest = w / tiles;
        l = rest % args.L;
        const int z = rest / args.L;
        plane = z / args.C;
        c = z % args.C;
        if ((plane ? args.out[1] : args.out[0]) == nullptr) return false;
        return !(args.accept && args.accept[c] == 0);  // rejected segment: left to a dense prefill
    };

    if (threadIdx.x == 0) {
        mbar_init(&afull, 1);
        mbar_init(&ascaled, kApEpi / 32);
        mbar_init(&adone, 1);
        mbar_init(&mdrain, 1);
        for (int i = 0; i < NX; ++i) {
            mbar_init(&xfull[i], 1);
            mbar_init(&xdone[i], kApEpi / 32);
            mbar_init(&xempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kApEpi / 32);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], 1);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 2 * GD);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 streams A and the x slabs, lane 1 the Bt ring (independent waits); the
        // rings run on across the units of this CTA
        if (lane == 0) {
            prefetch_tensormap(&tm_x0);
            prefetch_tensormap(&tm_x1);
            prefetch_tensormap(&tm_o0);
            prefetch_tensormap(&tm_o1);
            prefetch_tensormap(&tm_a0);
            prefetch_tensormap(&tm_a1);
            prefetch_tensormap(&tm_b0);
            prefetch_tensormap(&tm_b1);
            int it = 0, xn = 0;  // units; x slabs armed
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* mx = plane ? &tm_x1 : &tm_x0;
                const int t0 = tile * kAnRows;
                bool ok = true;
                for (int h = 0; h < H; ++h) {
                    const int hg = it * H + h, xi = hg % NX;
                    if (hg >= NX && !mbar_wait(&xempty[xi], (unsigned)(hg / NX - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&xfull[xi], (unsigned)K::kXBytes);
                    for (int b = 0; b < D / 64; ++b)
                        tma_load_4d(xs + xi * K::kXBytes + b * (kAnRows * 128), mx, h * D + 64 * b, t0, l, c, &xfull[xi]);
                    ++xn;
                }
                if (!ok) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                ++it;
            }
            if (anchor_vload(&abort_flag)) drain_ring(xfull, NX, xn);
        } else if (lane == 2) {
            // the A tiles of each unit, as soon as the previous unit's MMAs have read theirs
            int it = 0, an = 0;  // units; A loads armed
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* ma = plane ? &tm_a1 : &tm_a0;
                const int t0 = tile * kAnRows;
                if (it > 0 && !mbar_wait(&adone, (unsigned)(it - 1) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                mbar_arrive_expect_tx(&afull, (unsigned)(V * K::kABytes));
                for (int v = 0; v < V; ++v)
                    tma_load_2d(asm_ + v * K::kABytes, ma, 0, ((c * V + v) * args.L + l) * args.n + t0, &afull);
                ++an;
                ++it;
            }
            if (anchor_vload(&abort_flag)) drain_ring(&afull, 1, an);
        } else if (lane == 1) {
            int bn = 0, e = 0;  // Bt tiles armed; ring slot of the next
            unsigned ph = 0;     // phase parity of that slot's next fill
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* mb = plane ? &tm_b1 : &tm_b0;
                bool ok = true;
                // rows g * GD .. of each anchor's Bt (a short last group reads rows it does
                // not use: the next anchor's, or zero fill past the end)
                for (int g = 0; ok && g < groups && !anchor_vload(&abort_flag); ++g)
                    for (int v = 0; v < V; ++v) {
                        if (bn >= NB && !mbar_wait(&bempty[e], ph ^ 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&bfull[e], (unsigned)bslot);
                        tma_load_2d(bs + e * bslot, mb, 0, ((c * V + v) * args.L + l) * F + g * GD, &bfull[e]);
                        ++bn;
                        if (++e == NB) e = 0, ph ^= 1u;
                    }
                if (!ok) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
            }
            if (anchor_vload(&abort_flag)) drain_ring(bfull, NB, bn);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = true;
            int it = 0, gg = 0, e = 0;  // units; groups issued; Bt ring slot of the next
            unsigned bph = 0;           // its fill's phase parity
            const uint64_t a_first = tc_smem_desc(asm_, 16, 8 * K::kRowBytes, K::kLayout);
            const uint64_t b_first = tc_smem_desc(bs, 16, 8 * K::kRowBytes, K::kLayout);
            for (int w = blockIdx.x; ok && w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                if (!mbar_wait(&ascaled, (unsigned)it & 1u)) {
                    ok = false;
                    break;
                }
                for (int g = 0; ok && g < groups && !anchor_vload(&abort_flag); ++g, ++gg) {
                    const int a = gg & 1;
                    const int hn = H - g * G < G ? H - g * G : G;  // heads of this group
                    const uint32_t idesc = tc_idesc_bf16(kAnRows, hn * D);
                    if (gg >= 2 && !mbar_wait(&tempty[a], (unsigned)((gg >> 1) & 1) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors advance by 16-byte units (shared addresses stay below 256 KB)
                    uint64_t a_desc = a_first;
                    for (int v = 0; v < V; ++v) {
                        if (!mbar_wait(&bfull[e], bph)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t b_desc = b_first + (uint64_t)((e * bslot) >> 4);
#pragma unroll
                        for (int kk = 0; kk < R / 16; ++kk)
                            tc_mma_bf16(tmem + a * GD, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (v > 0 || kk > 0) ? 1u : 0u);
                        tc_commit(&bempty[e]);
                        if (++e == NB) e = 0, bph ^= 1u;
                        a_desc += (uint64_t)(K::kABytes >> 4);
                    }
                    if (ok) tc_commit(&tfull[a]);
                }
                tc_commit(&adone);  // this unit's MMAs are done with its A tiles
                ++it;
            }
            if (!ok) atomicOr(&abort_flag, 1);
            // every MMA issued has completed before the tensor memory is released
            tc_commit(&mdrain);
            mbar_wait(&mdrain, 0u);
        }
    } else if (warp == kApThreads / 32 - 1) {
        // ------------------------------------------------------------ TMA stores
        // each finished slab goes out, and is freed for the next load once read
        if (lane == 0) {
            int it = 0;
            for (int w = blockIdx.x; w < units && !anchor_vload(&abort_flag); w += gridDim.x) {
                int tile, l, plane, c;
                if (!unit_of(w, tile, l, plane, c)) continue;
                const CUtensorMap* mo = plane ? &tm_o1 : &tm_o0;
                const int t0 = tile * kAnRows;
                bool ok = true;
                for (int h = 0; h < H; ++h) {
                    const int hx = it * H + h, xi = hx % NX;
                    if (anchor_vload(&abort_flag) || !mbar_wait(&xdone[xi], (unsigned)(hx / NX) & 1u)) {
                        ok = false;
                        break;
                    }
                    unsigned char* slab = xs + xi * K::kXBytes;
                    for (int b = 0; b < D / 64; ++b)
                        tma_store_4d(mo, slab + b * (kAnRows * 128), h * D + 64 * b, t0, l, c);
                    bulk_commit();
                    bulk_wait_read<0>();
                    mbar_arrive(&xempty[xi]);
                }
                if (!ok) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                ++it;
            }
            bulk_wait<0>();
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // A warp that meets a failed wait skips the rest of the unit; all 256 threads meet
        // once per unit at the barrier that decides whether to go on.
        const int ew = warp - 2;             // 0..7
        const int wq = warp & 3;             // TMEM lane quarter of this warp
        const int half = ew >> 2;            // which half of a head's rotation pairs
        const int m = 32 * wq + lane;        // tile row
        const int et = threadIdx.x - 64;     // 0..255
        const int i0 = half * K::kPairs;     // first rotation pair (dims i0.., D/2 + i0..)
        bool ok = true;
        int it = 0, gg = 0;
        for (int w = blockIdx.x; w < units; w += gridDim.x) {
            int tile, l, plane, c;
            if (!unit_of(w, tile, l, plane, c)) continue;
            // the previous unit is done with the angle table; leave together on abort
            if (bar_any<1, kApEpi>(!ok || anchor_vload(&abort_flag))) break;
            const int t0 = tile * kAnRows;
            const bool row_ok = t0 + m < args.n;
            if (plane == 0)
                for (int i = et; i < D / 2; i += kApEpi) {
                    float cs, sn;
                    rope_cos_sin(args.delta[c], th.theta[i], &cs, &sn);
                    tab[i] = make_float2(cs, sn);
                }
            // scale each anchor's A tile row by the token's weight (bf16, in place: the swizzle
            // only permutes 16-byte pieces within the row).  Lane i of the warp holds the
            // weights of row 32 wq + i; in step k the warp scales the 32 consecutive 16-byte
            // pieces [32 k, 32 k + 32) of its 32 rows (conflict-free), taking each piece's
            // weight from its row's lane; the two warps of a lane quarter take alternate
            // steps.  The wait's outcome is made warp-uniform for the shuffles.
            // the row's weights, loaded while the A tiles are still on their way
            const float* wr = (plane ? args.w[1] : args.w[0]) + (((long long)c * args.L + l) * args.n + (row_ok ? t0 + m : 0)) * V;
            float wmine[kAnMaxAnchors];
#pragma unroll
            for (int v = 0; v < kAnMaxAnchors; ++v) wmine[v] = (v < V && row_ok) ? wr[v] : 0.f;
            if (__all_sync(0xffffffffu, mbar_wait(&afull, (unsigned)it & 1u))) {
                constexpr int kPieces = K::kRowBytes / 16;  // 16-byte pieces per row (2, 4 or 8)
#pragma unroll
                for (int v = 0; v < kAnMaxAnchors; ++v) {
                    if (v >= V) break;
                    unsigned char* at = asm_ + v * K::kABytes + (32 * wq) * K::kRowBytes;
#pragma unroll
                    for (int k = half; k < kPieces; k += 2) {
                        const int pc = 32 * k + lane, row = pc / kPieces;  // row within the warp's 32
                        const float wv = __shfl_sync(0xffffffffu, wmine[v], row);
                        uint4* pp = reinterpret_cast<uint4*>(at + pc * 16);
                        float f[8];
                        unpack8(*pp, f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) f[q] *= wv;
                        *pp = pack8(f);
                    }
                }
            } else {
                ok = false;
                atomicOr(&abort_flag, 1);
            }
            fence_proxy_async_smem();  // generic writes of A -> read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&ascaled);
            asm volatile("bar.sync 1, 256;" ::: "memory");  // the angle table is complete
            for (int g = 0; ok && g < groups; ++g, ++gg) {
                const int a = gg & 1;
                const int hn = H - g * G < G ? H - g * G : G;
                if (anchor_vload(&abort_flag) || !__all_sync(0xffffffffu, mbar_wait(&tfull[a], (unsigned)(gg >> 1) & 1u))) {
                    ok = false;
                    atomicOr(&abort_flag, 1);
                    break;
                }
                tc_fence_after();
                for (int hl = 0; hl < hn; ++hl) {
                    const int h = g * G + hl, hx = it * H + h, xi = hx % NX;
                    if (anchor_vload(&abort_flag) ||
                        !__all_sync(0xffffffffu, mbar_wait(&xfull[xi], (unsigned)(hx / NX) & 1u))) {
                        ok = false;
                        atomicOr(&abort_flag, 1);
                        break;
                    }
                    unsigned char* slab = xs + xi * K::kXBytes;
                    // this thread's rotation pairs of head h: dims i0 .. i0 + kPairs and their
                    // partners D/2 + i0 ..
                    const uint32_t tb = tmem + ((uint32_t)(32 * wq) << 16) + a * GD + hl * D;
                    uint32_t lo[K::kPairs], hi[K::kPairs];
                    if constexpr (K::kPairs == 32) {
                        tmem_ld32(tb + i0, lo);
                        tmem_ld32(tb + D / 2 + i0, hi);
                    } else {
                        tmem_ld16(tb + i0, lo);
                        tmem_ld16(tb + D / 2 + i0, hi);
                    }
                    tmem_wait_ld();
                    if (hl == hn - 1) {
                        // the group's accumulators are all in registers: free the slot
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[a]);
                    }
#pragma unroll
                    for (int q = 0; q < K::kPairs / 8; ++q) {
                        const int f0 = i0 + 8 * q, f1 = D / 2 + f0;  // first dims of the two pieces
                        uint4* p0 = reinterpret_cast<uint4*>(slab + (f0 / 64) * (kAnRows * 128) + m * 128 +
                                                             ((((f0 % 64) / 8) ^ (m & 7)) << 4));
                        uint4* p1 = reinterpret_cast<uint4*>(slab + (f1 / 64) * (kAnRows * 128) + m * 128 +
                                                             ((((f1 % 64) / 8) ^ (m & 7)) << 4));
                        float x0[8], x1[8];
                        unpack8(*p0, x0);
                        unpack8(*p1, x1);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float y0 = x0[e], y1 = x1[e];
                            if (plane == 0) {
                                const float2 cs = tab[f0 + e];
                                y0 = __fmaf_rn(x0[e], cs.x, __fmul_rn(x1[e], -cs.y));
                                y1 = __fmaf_rn(x1[e], cs.x, __fmul_rn(x0[e], cs.y));
                            }
                            x0[e] = y0 + __uint_as_float(lo[8 * q + e]);
                            x1[e] = y1 + __uint_as_float(hi[8 * q + e]);
                        }
                        *p0 = pack8(x0);
                        *p1 = pack8(x1);
                    }
                    fence_proxy_async_smem();  // epilogue writes -> TMA store reads
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&xdone[xi]);
                }
            }
            ++it;
        }
    }
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(&g_status_anchor, FLAG_TIMEOUT);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 2 * GD);
}

// ------------------------------------------------------------------ host side

// Tensor map of a bf16 plane view (dims: row elements, tokens, layers, chunks) with a
// (box_inner x 128 rows) box.
static cudaError_t anchor_plane_map(CUtensorMap* map, const void* base, const Plane& p, uint32_t box_inner,
                                    CUtensorMapSwizzle sw) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const long long row = (long long)p.heads * p.dim;
    cuuint64_t dims[4] = {(cuuint64_t)row, (cuuint64_t)p.tokens, (cuuint64_t)p.layers, (cuuint64_t)p.chunks};
    long long st = p.tokens > 1 ? p.st : row;
    long long sl = p.layers > 1 ? p.sl : st * p.tokens;
    long long sc = p.chunks > 1 ? p.sc : sl * p.layers;
    cuuint64_t strides[3] = {(cuuint64_t)(2 * st), (cuuint64_t)(2 * sl), (cuuint64_t)(2 * sc)};
    cuuint32_t box[4] = {box_inner, (cuuint32_t)kAnRows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of a factor viewed as [rows][r] bf16 with an (r x box_rows) box, swizzled
// by the row's byte length.
static cudaError_t anchor_factor_map(CUtensorMap* map, const void* base, long long rows, int r, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {(cuuint64_t)r, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)r * 2};
    cuuint32_t box[2] = {(cuuint32_t)r, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(r * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Static shared memory of the kernels, kept out of the dynamic budget.
constexpr int kAdStaticBytes = 2 * 1024;
constexpr int kApStaticBytes = 2 * 1024;

struct AdShape {
    int nb, nx, smem;
};

// After the A tiles and the row sums (one array, or two with the gate's): as many x
// buffers (up to 4) as leave room for at least 8 Bt entries (or 2 x buffers, or 1 when
// 2 leave no room for 2 entries), then the Bt ring takes the rest (up to 16).
static bool ad_shape(int V, int r, AdShape* s, int sum_arrays = 1) {
    const int row = 2 * r;
    const int abytes = kAnRows * row, bbytes = kAdCols * row, sums = sum_arrays * V * kAdEpi * (int)sizeof(float);
    const int room = kAnSmemLimit - kAdStaticBytes - 1024 - V * abytes - sums;
    for (s->nx = kAdMaxX; s->nx > 2 && room - s->nx * kAdXBytes < 8 * bbytes; --s->nx) {
    }
    if (room - s->nx * kAdXBytes < 2 * bbytes) s->nx = 1;
    s->nb = (room - s->nx * kAdXBytes) / bbytes;
    if (s->nb > kAdMaxB) s->nb = kAdMaxB;
    s->smem = 1024 + V * abytes + s->nx * kAdXBytes + s->nb * bbytes + sums;
    return V >= 1 && V <= kAnMaxAnchors && s->nb >= 2;
}

struct ApShape {
    int nb, nx, g, smem;
};

// Heads per MMA group 256 / D (N = 256 accumulator columns), halved while there are
// fewer heads or the rings do not fit; x slabs 3 with at least 3 Bt entries, else 2
// with at least 4 (one head per group: 2 slabs and 2 entries at least).
static bool ap_shape(int V, int r, int D, int H, ApShape* s) {
    const int row = 2 * r;
    const int abytes = kAnRows * row, xbytes = kAnRows * D * 2;
    const int base = kAnSmemLimit - kApStaticBytes - 1024 - V * abytes;
    for (s->g = 256 / D;; s->g /= 2) {
        const int bslot = s->g * D * row;
        bool fit = false;
        for (s->nx = kApMaxX; s->nx >= 2 && !fit; --s->nx) {
            const int budget = base - s->nx * xbytes;
            s->nb = budget > 0 ? budget / bslot : 0;
            if (s->nb > kApMaxB) s->nb = kApMaxB;
            fit = s->nb >= (s->nx == 3 ? 3 : 4);
            if (fit) break;
        }
        if (fit && s->g <= H) break;
        if (s->g == 1) {
            s->nx = 2;
            s->nb = base - 2 * xbytes > 0 ? (base - 2 * xbytes) / bslot : 0;
            if (s->nb > kApMaxB) s->nb = kApMaxB;
            break;
        }
    }
    s->smem = 1024 + V * abytes + s->nx * xbytes + s->nb * s->g * D * row;
    return V >= 1 && V <= kAnMaxAnchors && s->nb >= 2;
}

bool anchor_shape_ok(int anchors, int rank, int head_dim) {
    AdShape a;
    ApShape b;
    return ad_shape(anchors, rank, &a, 2) && (head_dim <= 0 || ap_shape(anchors, rank, head_dim, 1, &b));
}

size_t anchor_gate_workspace_bytes(const kvfix_kv_desc& d, int anchors, int prefix) {
    const long long tiles = (prefix + kAnRows - 1) / kAnRows;
    return (size_t)d.chunks * d.layers * tiles * anchors * sizeof(float);
}

template <int R, int MODE>
static cudaError_t launch_dist(const CUtensorMap* mx, const CUtensorMap* ma, const CUtensorMap* mb, AdArgs& args,
                               int planes, cudaStream_t s) {
    AdShape sh;
    if (!ad_shape(args.V, R, &sh, MODE == kAdBoth ? 2 : 1)) return cudaErrorInvalidValue;
    args.nb = sh.nb;
    args.nx = sh.nx;
    cudaError_t e = cudaFuncSetAttribute(anchor_dist_kernel<R, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (the shared-memory rings allow no second) walks the units
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long units = (long long)args.tiles * args.L * planes * args.C;
    if (units == 0) return cudaSuccess;
    dim3 grid((unsigned)(units < nsm ? units : (nsm > 0 ? nsm : 1)));
    anchor_dist_kernel<R, MODE><<<grid, kAdThreads, sh.smem, s>>>(mx[0], mx[1], ma[0], ma[1], mb[0], mb[1], args);
    return cudaGetLastError();
}

template <int R, int MODE>
static cudaError_t dist_maps_and_launch(const uint16_t* const* x, const Plane& p, const uint16_t* const* ac,
                                        const uint16_t* const* bct, AdArgs& args, int planes, cudaStream_t s) {
    CUtensorMap mx[2], ma[2], mb[2];
    cudaError_t e;
    const long long arows = (long long)args.C * args.V * args.L * args.n;
    const long long brows = (long long)args.C * args.V * args.L * args.F;
    for (int q = 0; q < 2; ++q) {
        const int src = q < planes ? q : 0;
        if ((e = anchor_plane_map(&mx[q], x[src], p, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
        if ((e = anchor_factor_map(&ma[q], ac[src], arows, R, kAnRows)) != cudaSuccess) return e;
        if ((e = anchor_factor_map(&mb[q], bct[src], brows, R, kAdCols)) != cudaSuccess) return e;
    }
    return launch_dist<R, MODE>(mx, ma, mb, args, planes, s);
}

cudaError_t launch_anchor_gate(const uint16_t* v_src, const kvfix_kv_desc& d, const uint16_t* ac,
                               const uint16_t* bct, int V, int r, int k, double T, double tau, double* dist,
                               double* g, double* hbar, int32_t* accept, void* workspace, cudaStream_t s) {
    Plane p = plane_of(d);
    if (p.chunks == 0) return cudaSuccess;
    AdArgs args = {};
    args.V = V;
    args.L = p.layers;
    args.n = p.tokens;
    args.F = p.heads * p.dim;
    args.C = p.chunks;
    args.rows = k;
    args.tiles = (k + kAnRows - 1) / kAnRows;
    args.inv_T = (float)(1.0 / T);
    args.partial = static_cast<float*>(workspace);
    const uint16_t* xs[1] = {v_src};
    const uint16_t* as[1] = {ac};
    const uint16_t* bs[1] = {bct};
    cudaError_t e;
    if (r == 16) e = dist_maps_and_launch<16, kAdGate>(xs, p, as, bs, args, 1, s);
    else if (r == 32) e = dist_maps_and_launch<32, kAdGate>(xs, p, as, bs, args, 1, s);
    else e = dist_maps_and_launch<64, kAdGate>(xs, p, as, bs, args, 1, s);
    if (e != cudaSuccess) return e;
    anchor_gate_kernel<<<p.chunks, 32 * kAnMaxAnchors, 0, s>>>(args.partial, V, p.layers, args.tiles, T, tau, dist, g, hbar, accept);
    return cudaGetLastError();
}

template <int D, int R>
static cudaError_t launch_apply(const uint16_t* const* x, const Plane& p, uint16_t* const* out, const Plane& op,
                                const uint16_t* const* ad, const uint16_t* const* bdt, ApArgs& args,
                                const RopeTheta& th, cudaStream_t s) {
    ApShape sh;
    if (!ap_shape(args.V, R, D, args.H, &sh)) return cudaErrorInvalidValue;
    args.nb = sh.nb;
    args.nx = sh.nx;
    args.G = sh.g;
    CUtensorMap mx[2], mo[2], ma[2], mb[2];
    cudaError_t e;
    const long long arows = (long long)args.C * args.V * args.L * args.n;
    const long long brows = (long long)args.C * args.V * args.L * args.H * D;
    for (int q = 0; q < 2; ++q) {
        if ((e = anchor_plane_map(&mx[q], x[q], p, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
        if ((e = anchor_plane_map(&mo[q], out[q], op, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
        if ((e = anchor_factor_map(&ma[q], ad[q], arows, R, kAnRows)) != cudaSuccess) return e;
        if ((e = anchor_factor_map(&mb[q], bdt[q], brows, R, (uint32_t)(sh.g * D))) != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(anchor_apply_kernel<D, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, sh.smem);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, anchor_apply_kernel<D, R>, kApThreads, sh.smem)) != cudaSuccess)
        return e;
    const long long units = (long long)((args.n + kAnRows - 1) / kAnRows) * args.L * 2 * args.C;
    if (units == 0) return cudaSuccess;
    const long long slots = (long long)(nsm > 0 ? nsm : 1) * (per_sm > 0 ? per_sm : 1);
    dim3 grid((unsigned)(units < slots ? units : slots));
    anchor_apply_kernel<D, R><<<grid, kApThreads, sh.smem, s>>>(mx[0], mx[1], mo[0], mo[1], ma[0], ma[1], mb[0],
                                                                 mb[1], args, th);
    return cudaGetLastError();
}

cudaError_t launch_anchor_correct(const AnchorPlanes& pl, const kvfix_kv_desc& d, const kvfix_kv_desc& od, int V,
                                  int r, double T, const int32_t* delta, const RopeTheta& th,
                                  const int32_t* accept, cudaStream_t s, const AnchorGateOut* gate) {
    Plane p = plane_of(d), op = plane_of(od);
    if (p.chunks == 0 || p.layers == 0 || p.tokens == 0) return cudaSuccess;
    AdArgs args = {};
    args.V = V;
    args.L = p.layers;
    args.n = p.tokens;
    args.F = p.heads * p.dim;
    args.C = p.chunks;
    args.rows = p.tokens;
    args.tiles = (p.tokens + kAnRows - 1) / kAnRows;
    args.inv_T = (float)(1.0 / T);
    args.w[0] = pl.w[0];
    args.w[1] = pl.w[1];
    args.accept = accept;
    cudaError_t e;
    if (gate) {
        // the gate from the value plane's reconstructions of the same pass
        args.partial = static_cast<float*>(gate->workspace);
        args.gate_rows = gate->k;
        if (r == 16) e = dist_maps_and_launch<16, kAdBoth>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        else if (r == 32) e = dist_maps_and_launch<32, kAdBoth>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        else e = dist_maps_and_launch<64, kAdBoth>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        if (e != cudaSuccess) return e;
        anchor_gate_kernel<<<p.chunks, 32 * kAnMaxAnchors, 0, s>>>(args.partial, V, p.layers, args.tiles, gate->T,
                                                                    gate->tau, gate->d, gate->g, gate->hbar,
                                                                    gate->accept);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        accept = gate->accept;
    } else {
        if (r == 16) e = dist_maps_and_launch<16, kAdWeights>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        else if (r == 32) e = dist_maps_and_launch<32, kAdWeights>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        else e = dist_maps_and_launch<64, kAdWeights>(pl.src, p, pl.ac, pl.bct, args, 2, s);
        if (e != cudaSuccess) return e;
    }
    ApArgs ap = {};
    ap.V = V;
    ap.L = p.layers;
    ap.n = p.tokens;
    ap.H = p.heads;
    ap.C = p.chunks;
    ap.w[0] = pl.w[0];
    ap.w[1] = pl.w[1];
    ap.accept = accept;
    ap.delta = delta;
    ap.out[0] = pl.out[0];
    ap.out[1] = pl.out[1];
    if (p.dim == 128) {
        if (r == 16) return launch_apply<128, 16>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
        if (r == 32) return launch_apply<128, 32>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
        return launch_apply<128, 64>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
    }
    if (r == 16) return launch_apply<64, 16>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
    if (r == 32) return launch_apply<64, 32>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
    return launch_apply<64, 64>(pl.src, p, pl.out, op, pl.ad, pl.bdt, ap, th, s);
}

}  // namespace kvfix
