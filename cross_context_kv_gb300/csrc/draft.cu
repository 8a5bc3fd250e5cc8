// draft.cu -- kvfix_draft_rank: rank cached rows by the softmax attention mass of the
// draft queries, keep the best k rows, optionally overwrite them with fresh rows.
//
// Method: Budgeted Cache Repair, section 3 ("The repair": row score a_j summed over
// layers after the first, steps and heads of softmax(Q K~^T / sqrt(d_head))), App. B
// Algorithm 2 (grouped-query keys expanded to query heads) and Algorithm 1 (the
// selected rows' K and V are overwritten before use); KVCMAS Eq. 3.
//
// Pipeline (one unit = chunk, layer >= layer_begin, KV head; its G = steps x
// q_heads/kv_heads <= 16 query rows share the unit's keys):
//   1. rank:    one cluster per unit: tensor-core QK^T per 128-key tile with the logits
//               kept in tensor memory, softmax statistics combined over the cluster,
//               each key's mass sum_q exp(z - max_q) / sum_q to the workspace [unit][n];
//   2. accum:   per key, the masses of the chunk's units added in a fixed order
//               (layer-major, then head) with compensated float sums;
//   3. select:  top-k of the double scores (ties to the lower index);
//   4. repair:  copy the selected rows of every layer and head from the fresh planes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cooperative_groups.h>

#include "softmax.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace kvfix {

static __device__ unsigned int g_status_draft;

unsigned read_status_draft(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_draft, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_draft, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

// One unit = (chunk, layer >= layer_begin, KV head): its G <= 16 query rows (draft steps
// x query heads of the group) and its n keys.  A cluster of 8 CTAs takes a unit; CTA k
// takes key tiles [k*tpc, (k+1)*tpc) of 128 keys:
//   warp 0      TMA producer: key tiles (128 keys x D, two 64-column boxes, 128-byte
//               swizzle) into a 3-stage ring;
//   warp 1      tcgen05.mma M=128 (keys) x N=16 (queries) x K=D; the logits of tile t stay
//               in tensor memory, columns [16t, 16t+16), so no logit goes to HBM;
//   warps 2..5  softmax: per query, max and sum of exp over the CTA's keys (read back
//               from TMEM), combined over the cluster through distributed shared memory
//               in rank order; then each key's mass sum_q exp(z - max_q) / sum_q.
// The per-key masses go to the workspace [unit][n]; a second kernel adds them over the
// units of a chunk (layer-major, then head) in a fixed order as compensated float pairs
// (about 48 significant bits), returned as doubles.
constexpr int kDcCluster = 8;
constexpr int kDcThreads = 192;
constexpr int kDcStages = 3;
constexpr int kDcRows = 128;   // keys per tile (MMA M)
constexpr int kDcQ = 16;       // query rows per unit, padded (MMA N)
// The softmax works in base 2: exp(z - m) = 2^((z - m) log2 e), with the logits scaled by
// log2 e once, so each term is one exp2f.
constexpr float kLog2e = 1.4426950408889634f;

static long long dc_units(const kvfix_kv_desc& d, int layer_begin) {
    const long long nl = d.layers > layer_begin ? d.layers - layer_begin : 0;
    return (long long)d.chunks * nl * d.kv_heads;
}

size_t draft_workspace_bytes(const kvfix_kv_desc& d, int layer_begin) {
    return ((sizeof(float) * (size_t)dc_units(d, layer_begin) * (size_t)d.tokens + 255) / 256) * 256;
}

// Tiles per CTA such that the CTA's logits fit the 512 TMEM columns.
static int dc_tiles_per_cta(int n) {
    const int tiles = (n + kDcRows - 1) / kDcRows;
    return (tiles + kDcCluster - 1) / kDcCluster;
}

static int pow2_at_least(int x) {
    int c = 32;
    while (c < x) c <<= 1;
    return c;
}

struct DcArgs {
    const uint16_t* q;   // [C][L][steps][Hq][D]
    float* contrib;      // [units][n]
    int L, n, H, steps, q_heads, layer_begin, G, tpc, tmem_cols;
};

// Shared memory is padded to at least 80 KB so that at most two CTAs share an SM: each
// holds up to 256 TMEM columns, and two never exceed the SM's 512 (an allocation that
// had to wait for another cluster's CTA could otherwise deadlock the clusters).
template <int D>
struct DcCfg {
    static constexpr int kTile = kDcRows * D * 2;
    static constexpr int kQBytes = kDcQ * D * 2;
    static constexpr int kNeed = 1024 + kDcStages * kTile + kQBytes;
    static constexpr int kSmem = kNeed > 80 * 1024 ? kNeed : 80 * 1024;
};

template <int D>
__global__ void __cluster_dims__(kDcCluster, 1, 1) __launch_bounds__(kDcThreads, 1)
draft_cluster_kernel(const __grid_constant__ CUtensorMap tm_k, DcArgs args) {
    using C = DcCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t full[kDcStages], empty[kDcStages], done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float red_m[4][kDcQ], red_s[4][kDcQ];
    __shared__ float cta_m[kDcQ], cta_s[kDcQ], fin_m[kDcQ], fin_inv[kDcQ];
    cg::cluster_group cluster = cg::this_cluster();
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* qsm = smem + kDcStages * C::kTile;  // Q, K-major canonical, no swizzle
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster.block_rank();
    const long long unit = blockIdx.y;
    const int nl = args.L - args.layer_begin;
    const int kvh = (int)(unit % args.H);
    const int l = args.layer_begin + (int)((unit / args.H) % nl);
    const int c = (int)(unit / ((long long)args.H * nl));
    const int n = args.n;
    const int tiles = (n + kDcRows - 1) / kDcRows;
    const int tile0 = rank * args.tpc;
    const int ntiles = max(0, min(args.tpc, tiles - tile0));
    const int group = args.q_heads / args.H;

    // Q rows i = t*group + m  <->  q[c][l][t][kvh*group + m], zero-padded to 16 rows;
    // element (i, e) at (i%8)*16 + (i/8)*SBO + (e/8)*128 + (e%8)*2 with SBO = (D/8)*128.
    for (int idx = threadIdx.x; idx < kDcQ * D; idx += kDcThreads) {
        const int i = idx / D, e = idx % D;
        uint16_t v = 0;
        if (i < args.G) {
            const int t = i / group, m = i % group;
            v = args.q[((((long long)c * args.L + l) * args.steps + t) * args.q_heads + kvh * group + m) * D + e];
        }
        *reinterpret_cast<uint16_t*>(qsm + (i % 8) * 16 + (i / 8) * (D / 8) * 128 + (e / 8) * 128 + (e % 8) * 2) = v;
    }
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int st = 0; st < kDcStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        mbar_init(&done, 1);
        fence_mbar_init();
        abort_flag = 0;
        prefetch_tensormap(&tm_k);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, (uint32_t)args.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % kDcStages;
                if (i >= kDcStages && !mbar_wait(&empty[st], (unsigned)(i / kDcStages - 1) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                unsigned char* dst = smem + st * C::kTile;
                mbar_arrive_expect_tx(&full[st], C::kTile);
                for (int half = 0; half < D / 64; ++half)
                    tma_load_4d(dst + half * (kDcRows * 128), &tm_k, kvh * D + 64 * half, (tile0 + i) * kDcRows, l,
                                c, &full[st]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc_bf16(kDcRows, kDcQ);
            bool ok = true;
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % kDcStages;
                if (!mbar_wait(&full[st], (unsigned)(i / kDcStages) & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const unsigned char* kt = smem + st * C::kTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t adesc = tc_smem_desc(kt + (kk / 4) * (kDcRows * 128) + 32 * (kk % 4), 16, 1024, 2);
                    const uint64_t bdesc = tc_smem_desc(qsm + 256 * kk, 128, (D / 8) * 128, 0);
                    tc_mma_bf16(tmem + kDcQ * i, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(&empty[st]);  // the stage is free once these MMAs have read it
            }
            if (!ok) atomicOr(&abort_flag, 1);
            tc_commit(&done);  // every logit of this CTA is in TMEM
        }
    } else {
        // ------------------------------------------------------------ softmax
        // one pass over the CTA's logits, tile by tile: per query row the running maximum
        // and rescaled sum (softmax.cuh); then the warp's and the CTA's pairs
        const int wq = warp & 3, ew = warp - 2;
        const int key_in_tile = 32 * wq + lane;
        const float scale = rsqrtf((float)D) * kLog2e;  // logits in base-2 units
        const bool ok = mbar_wait(&done, 0u);
        if (!ok) atomicOr(&abort_flag, 1);
        tc_fence_after();
        float mx[kDcQ], sm[kDcQ];
#pragma unroll
        for (int q = 0; q < kDcQ; ++q) {
            mx[q] = -INFINITY;
            sm[q] = 0.f;
        }
        for (int i = 0; i < ntiles && ok; ++i) {
            const int key = (tile0 + i) * kDcRows + key_in_tile;
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * wq) << 16) + kDcQ * i, v);
            tmem_wait_ld();
            if (key < n) {
#pragma unroll
                for (int q = 0; q < kDcQ; ++q) online_add(mx[q], sm[q], __uint_as_float(v[q]) * scale);
            }
        }
#pragma unroll
        for (int q = 0; q < kDcQ; ++q) warp_combine(mx[q], sm[q]);
        if (lane == 0)
#pragma unroll
            for (int q = 0; q < kDcQ; ++q) {
                red_m[ew][q] = mx[q];
                red_s[ew][q] = sm[q];
            }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (threadIdx.x - 64 < kDcQ) {
            const int q = threadIdx.x - 64;
            const float m4[4] = {red_m[0][q], red_m[1][q], red_m[2][q], red_m[3][q]};
            const float s4[4] = {red_s[0][q], red_s[1][q], red_s[2][q], red_s[3][q]};
            combine4(m4, s4, cta_m[q], cta_s[q]);
        }
    }
    // ---------------- cluster: combine the 8 CTAs' (max, sum) in rank order
    cluster.sync();
    if (threadIdx.x < kDcQ) {
        const int q = threadIdx.x;
        float m = -INFINITY;
        for (int k = 0; k < kDcCluster; ++k) m = fmaxf(m, cluster.map_shared_rank(cta_m, k)[q]);
        float ssum = 0.f;
        for (int k = 0; k < kDcCluster; ++k) {
            const float mk = cluster.map_shared_rank(cta_m, k)[q];
            const float sk = cluster.map_shared_rank(cta_s, k)[q];
            if (mk != -INFINITY) ssum += sk * exp2f(mk - m);
        }
        fin_m[q] = m;
        fin_inv[q] = ssum > 0.f ? 1.0f / ssum : 0.f;
    }
    cluster.sync();  // also: no CTA leaves while others still read its shared memory
    if (warp >= 2) {
        const int wq = warp & 3;
        const int key_in_tile = 32 * wq + lane;
        const float scale = rsqrtf((float)D) * kLog2e;  // logits in base-2 units
        float* out = args.contrib + unit * (long long)n;
        for (int i = 0; i < ntiles && !abort_flag; ++i) {
            const int key = (tile0 + i) * kDcRows + key_in_tile;
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * wq) << 16) + kDcQ * i, v);
            tmem_wait_ld();
            float acc = 0.f;
            for (int q = 0; q < args.G; ++q) acc += exp2f(__uint_as_float(v[q]) * scale - fin_m[q]) * fin_inv[q];
            if (key < n) out[key] = acc;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(&g_status_draft, FLAG_TIMEOUT);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, (uint32_t)args.tmem_cols);
}

// ---- 2. accum: sum of the per-unit masses, grid = (ceil(n/256), chunks) ----------------------------
// Units are added in order (layer-major, then head) as a compensated float pair: the
// running sum and its rounding errors (Knuth's TwoSum), so the result carries about 48
// significant bits, is the same on every run, and costs no double-precision arithmetic
// (weak on this part).  Eight masses are loaded before they are added.
constexpr int kAccThreads = 256;
constexpr int kAccBatch = 8;

__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x) {
    const float s = __fadd_rn(hi, x);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
    hi = s;
    lo = __fadd_rn(lo, err);
}

__global__ void __launch_bounds__(kAccThreads)
draft_accum_kernel(const float* __restrict__ contrib, int n, long long units_per_chunk, double* scores) {
    const int c = blockIdx.y;
    const int j = blockIdx.x * kAccThreads + threadIdx.x;
    if (j >= n) return;
    const float* p = contrib + (long long)c * units_per_chunk * n + j;
    float hi = 0.f, lo = 0.f;
    long long u = 0;
    for (; u + kAccBatch <= units_per_chunk; u += kAccBatch) {
        float v[kAccBatch];
#pragma unroll
        for (int q = 0; q < kAccBatch; ++q) v[q] = __ldg(p + (u + q) * n);
#pragma unroll
        for (int q = 0; q < kAccBatch; ++q) two_sum_acc(hi, lo, v[q]);
    }
    for (; u < units_per_chunk; ++u) two_sum_acc(hi, lo, __ldg(p + u * n));
    scores[(long long)c * n + j] = (double)hi + (double)lo;
}

// ---- 3. select (double keys) --------------------------------------------------------
constexpr int kSelThreads2 = 1024;
constexpr int kSelSmemKeys2 = 16384;

__device__ __forceinline__ unsigned long long ordered_f64(double f) {
    unsigned long long u = (unsigned long long)__double_as_longlong(f);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

__device__ int block_exclusive_scan2(int x, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) warp_sums[lane] = wi - ws;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    int ex = inc - x + warp_sums[warp];
    *total = warp_sums[32];
    __syncthreads();
    return ex;
}

// Radix select of the k largest 64-bit keys (ties to the lower index).
__global__ void __launch_bounds__(kSelThreads2)
select_f64_kernel(const double* __restrict__ scores, int n, int kk, int32_t* idx) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ unsigned hist[256];
    __shared__ int warp_sums[33];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_remaining;
    const int words = (n + 31) / 32;
    uint32_t* bits = reinterpret_cast<uint32_t*>(dyn);
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(dyn + ((sizeof(uint32_t) * words + 15) / 16) * 16);
    const bool cached = n <= kSelSmemKeys2;
    const long long c = blockIdx.x;
    const double* sc = scores + c * n;
    int32_t* out = idx + c * kk;
    const int tid = threadIdx.x;
    auto key_at = [&](int i) -> unsigned long long { return cached ? keys[i] : ordered_f64(sc[i]); };
    for (int w = tid; w < words; w += blockDim.x) bits[w] = 0u;
    if (cached)
        for (int i = tid; i < n; i += blockDim.x) keys[i] = ordered_f64(sc[i]);
    if (tid == 0) {
        s_prefix = 0ull;
        s_remaining = kk;
    }
    __syncthreads();
    if (kk <= 0) return;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        const unsigned long long prefix = s_prefix;
        const unsigned long long hi_mask = shift == 56 ? 0ull : ~((1ull << (shift + 8)) - 1ull);
        for (int i = tid; i < n; i += blockDim.x) {
            unsigned long long kv = key_at(i);
            if ((kv & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(unsigned)(kv >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            unsigned cnt[8];
            unsigned lsum = 0;
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
                cnt[qq] = hist[255 - 8 * tid - qq];
                lsum += cnt[qq];
            }
            unsigned inc = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (tid >= o) inc += y;
            }
            const unsigned before = inc - lsum;
            const unsigned rem = (unsigned)s_remaining;
            if (before < rem && rem <= inc) {
                unsigned acc = before;
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    if (acc < rem && rem <= acc + cnt[qq]) {
                        s_prefix = prefix | ((unsigned long long)(255 - 8 * tid - qq) << shift);
                        s_remaining = (int)(rem - acc);
                    }
                    acc += cnt[qq];
                }
            }
        }
        __syncthreads();
    }
    const unsigned long long T = s_prefix;
    const int need_eq = s_remaining;
    const int seg = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += (key_at(i) == T);
    int tot;
    int eq_before = block_exclusive_scan2(eq, warp_sums, &tot);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) {
        unsigned long long kv = key_at(i);
        bool take = kv > T;
        if (kv == T) {
            take = eq_before < need_eq;
            ++eq_before;
        }
        if (take) {
            atomicOr(&bits[i >> 5], 1u << (i & 31));
            ++cnt;
        }
    }
    int ob = block_exclusive_scan2(cnt, warp_sums, &tot);
    __syncthreads();
    for (int i = i0; i < i1; ++i)
        if ((bits[i >> 5] >> (i & 31) & 1u) && ob < kk) out[ob++] = i;
}

static cudaError_t encode_keys(CUtensorMap* map, const uint16_t* base, const Plane& p) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const long long row = (long long)p.heads * p.dim;
    cuuint64_t dims[4] = {(cuuint64_t)row, (cuuint64_t)p.tokens, (cuuint64_t)p.layers, (cuuint64_t)p.chunks};
    long long st = p.tokens > 1 ? p.st : row;
    long long sl = p.layers > 1 ? p.sl : st * p.tokens;
    long long sc = p.chunks > 1 ? p.sc : sl * p.layers;
    cuuint64_t strides[3] = {(cuuint64_t)(2 * st), (cuuint64_t)(2 * sl), (cuuint64_t)(2 * sc)};
    cuuint32_t box[4] = {64, (cuuint32_t)kDcRows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_draft_finish(const float* contrib, int chunks, int n, long long units_per_chunk, int k_rows,
                                int32_t* idx, double* scores, cudaStream_t s) {
    cudaError_t e;
    if (chunks == 0 || n == 0) return cudaSuccess;
    if (units_per_chunk == 0) {
        e = cudaMemsetAsync(scores, 0, sizeof(double) * (size_t)chunks * n, s);
        if (e != cudaSuccess) return e;
    } else {
        dim3 g3((n + kAccThreads - 1) / kAccThreads, chunks);
        draft_accum_kernel<<<g3, kAccThreads, 0, s>>>(contrib, n, units_per_chunk, scores);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (k_rows > 0) {
        const int words = (n + 31) / 32;
        size_t smem = ((sizeof(uint32_t) * words + 15) / 16) * 16 + (n <= kSelSmemKeys2 ? sizeof(unsigned long long) * n : 0);
        e = cudaFuncSetAttribute(select_f64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        select_f64_kernel<<<chunks, kSelThreads2, smem, s>>>(scores, n, k_rows, idx);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_draft(const uint16_t* k, const kvfix_kv_desc& d, const uint16_t* q, int steps,
                         int q_heads, int layer_begin, int k_rows, int32_t* idx, double* scores,
                         void* ws_ptr, cudaStream_t s) {
    Plane p = plane_of(d);
    const int n = p.tokens;
    const int nl = p.layers - layer_begin;
    const long long units_per_chunk = (long long)nl * p.heads;
    const long long units = units_per_chunk * p.chunks;
    cudaError_t e;
    if (p.chunks == 0 || n == 0) return cudaSuccess;
    if (units > 0) {
        if (units > 65535) return cudaErrorInvalidValue;
        CUtensorMap tk;
        if ((e = encode_keys(&tk, k, p)) != cudaSuccess) return e;
        DcArgs a;
        a.q = q;
        a.contrib = static_cast<float*>(ws_ptr);
        a.L = p.layers;
        a.n = n;
        a.H = p.heads;
        a.steps = steps;
        a.q_heads = q_heads;
        a.layer_begin = layer_begin;
        a.G = steps * (q_heads / p.heads);
        a.tpc = dc_tiles_per_cta(n);
        a.tmem_cols = pow2_at_least(kDcQ * a.tpc);
        if (a.tmem_cols > 256) return cudaErrorInvalidValue;  // n <= 16384
        dim3 grid(kDcCluster, (unsigned)units);
        if (p.dim == 128) {
            e = cudaFuncSetAttribute(draft_cluster_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DcCfg<128>::kSmem);
            if (e != cudaSuccess) return e;
            draft_cluster_kernel<128><<<grid, kDcThreads, DcCfg<128>::kSmem, s>>>(tk, a);
        } else {
            e = cudaFuncSetAttribute(draft_cluster_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DcCfg<64>::kSmem);
            if (e != cudaSuccess) return e;
            draft_cluster_kernel<64><<<grid, kDcThreads, DcCfg<64>::kSmem, s>>>(tk, a);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return launch_draft_finish(static_cast<const float*>(ws_ptr), p.chunks, n, units_per_chunk, k_rows, idx, scores, s);
}

// ---- 4. row repair: grid = (ceil(k/16), L, C) ----------------------------------------
constexpr int kRepThreads = 256;
constexpr int kRepRows = 16;

// idx holds `kk` entries per chunk; with counts, only the first counts[c] are rows.
__global__ void __launch_bounds__(kRepThreads)
row_repair_kernel(uint16_t* io, Plane p, const uint16_t* __restrict__ fresh, Plane fp,
                  const int32_t* __restrict__ idx, int kk, const int32_t* __restrict__ counts) {
    const int l = blockIdx.y, c = blockIdx.z;
    const int row8 = p.heads * p.dim / 8;
    const int i0 = blockIdx.x * kRepRows;
    const int used = counts ? min(kk, counts[c]) : kk;
    const int rows = min(kRepRows, used - i0);
    for (int it = threadIdx.x; it < rows * row8; it += kRepThreads) {
        const int i = i0 + it / row8, v = it % row8;
        const int j = idx[(long long)c * kk + i];
        if (j < 0 || j >= p.tokens) {
            if (v == 0) atomicOr(&g_status_draft, FLAG_BOUNDS);
            continue;
        }
        uint4 val = ld_stream(reinterpret_cast<const uint4*>(fresh + fp.row(c, l, j) + 8ll * v));
        st_stream(reinterpret_cast<uint4*>(io + p.row(c, l, j) + 8ll * v), val);
    }
}

cudaError_t launch_row_repair(uint16_t* io, const kvfix_kv_desc& d, const uint16_t* fresh,
                              const kvfix_kv_desc& fd, const int32_t* idx, int k_rows,
                              cudaStream_t s, const int32_t* counts) {
    Plane p = plane_of(d), fp = plane_of(fd);
    if (k_rows == 0 || p.layers == 0 || p.chunks == 0) return cudaSuccess;
    dim3 grid((k_rows + kRepRows - 1) / kRepRows, p.layers, p.chunks);
    row_repair_kernel<<<grid, kRepThreads, 0, s>>>(io, p, fresh, fp, idx, k_rows, counts);
    return cudaGetLastError();
}

}  // namespace kvfix
