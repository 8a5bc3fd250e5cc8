// layout.cu -- the rows a draft-scored repair recomputes, in the three layouts of Budgeted
// Cache Repair (kvfix_repair_layout), and the overwrite of a counted row list
// (kvfix_repair_rows).
//
// Method: Budgeted Cache Repair, section 3 "The layouts" (BCR-single: the best rows;
// BCR-chunk: fixed 64-token chunks, the best rho of them; BCR-grow: a span seeded on the
// best row, extended while a neighbour scores at least tau of the seed); App. A.2 "The
// policy" (a chunk is scored by the mean of its rows, a short trailing chunk by its own
// mean) and Table 8 (max(1, round(rho n_chunks)) chunks); App. B, Algorithm 1 (skip when
// M < 2B or rho M < B; round(rho M / B) chunks) and Algorithm 2 (chunk scores).
//
// One CTA per unit: the keys (row scores, or chunk means summed row by row in index
// order) sit in shared memory; an 8-bit radix search marks the best rows or chunks
// (ties to the lower index), and a block scan turns the row bitmap into the ascending
// row list.  The grow layout's walk is sequential by definition (each seed depends on the
// spans before it): the k best rows are sorted by (score desc, index asc) with a bitonic
// sort and one thread walks them with the scores and the bitmap in shared memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

static __device__ unsigned int g_status_layout;

unsigned read_status_layout(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_layout, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_layout, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

constexpr int kLayThreads = 1024;

struct LayoutArgs {
    int n, layout, B;
    int k;          // rows (single, grow)
    int c;          // chunks (chunk layout)
    int skipped;    // chunk layout: the skip rule fired
    double tau;
    int max_rows;
};

// Keys are kept as order-preserving integers (lay_ord below): the same comparisons as
// the doubles', done by the integer pipes.
// key order: a before b iff key[a] > key[b], or equal keys and a < b; -1 pads last
__device__ __forceinline__ bool lay_before(const unsigned long long* key, int a, int b) {
    if (a < 0) return false;
    if (b < 0) return true;
    const unsigned long long ka = key[a], kb = key[b];
    return ka > kb || (ka == kb && a < b);
}

// Exclusive scan of one int per thread over the block; *total receives the sum.
__device__ __forceinline__ int lay_scan(int x, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_sums[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int v = lane < nw ? warp_sums[lane] : 0, wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < nw) warp_sums[lane] = wi - v;
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    const int ex = inc - x + warp_sums[warp];
    *total = warp_sums[32];
    __syncthreads();
    return ex;
}

// Order-preserving map of a (non-NaN) double to an unsigned key: larger double, larger
// key; -0 is first made +0, so that equal doubles give equal keys.
__device__ __forceinline__ unsigned long long lay_ord(double x) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(x + 0.0);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double lay_unord(unsigned long long k) {
    const unsigned long long u = (k >> 63) ? (k & 0x7fffffffffffffffull) : ~k;
    return __longlong_as_double((long long)u);
}

// Marks in `cand` (bitmap over N keys, cleared) the m largest keys, ties to the lower
// index: an 8-bit radix search for the m-th largest key T, then every key above T and
// the first (in index order) of those equal to T.
__device__ void lay_top(const unsigned long long* key, int N, int m, uint32_t* cand, unsigned* hist, int* warp_sums,
                        unsigned long long* s_prefix, int* s_remaining) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        *s_prefix = 0ull;
        *s_remaining = m;
    }
    __syncthreads();
    if (m <= 0) return;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kLayThreads) hist[i] = 0u;
        __syncthreads();
        const unsigned long long prefix = *s_prefix;
        const unsigned long long hi_mask = shift == 56 ? 0ull : ~((1ull << (shift + 8)) - 1ull);
        for (int i = tid; i < N; i += kLayThreads) {
            const unsigned long long kv = key[i];
            if ((kv & hi_mask) == (prefix & hi_mask)) atomicAdd(&hist[(unsigned)(kv >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            // lane t holds bins 255-8t .. 248-8t (largest first)
            unsigned cnt[8], lsum = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                cnt[q] = hist[255 - 8 * tid - q];
                lsum += cnt[q];
            }
            unsigned inc = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (tid >= o) inc += y;
            }
            const unsigned before = inc - lsum, rem = (unsigned)*s_remaining;
            if (before < rem && rem <= inc) {
                unsigned acc = before;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (acc < rem && rem <= acc + cnt[q]) {
                        *s_prefix = prefix | ((unsigned long long)(255 - 8 * tid - q) << shift);
                        *s_remaining = (int)(rem - acc);
                    }
                    acc += cnt[q];
                }
            }
        }
        __syncthreads();
    }
    const unsigned long long T = *s_prefix;
    const int need_eq = *s_remaining;
    const int seg = (N + kLayThreads - 1) / kLayThreads;
    const int i0 = min(N, tid * seg), i1 = min(N, i0 + seg);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += key[i] == T;
    int tot;
    int eq_before = lay_scan(eq, warp_sums, &tot);
    for (int i = i0; i < i1; ++i) {
        const unsigned long long kv = key[i];
        bool take = kv > T;
        if (kv == T) take = eq_before++ < need_eq;
        if (take) atomicOr(&cand[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
}

// grid = units.  Dynamic shared memory: key double[N], candidate bitmap over N, row
// bitmap over n, order int[P] (grow layout only).
__global__ void __launch_bounds__(kLayThreads)
repair_layout_kernel(const double* __restrict__ scores, LayoutArgs a, int N, int P, int32_t* idx,
                     int32_t* counts) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ int warp_sums[33];
    __shared__ unsigned hist[256];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_remaining, s_chosen;
    const int n = a.n, words = (n + 31) / 32, cwords = (N + 31) / 32;
    unsigned long long* key = reinterpret_cast<unsigned long long*>(dyn);
    uint32_t* cand = reinterpret_cast<uint32_t*>(dyn + (size_t)8 * N);
    uint32_t* bits = cand + cwords;
    int* order = reinterpret_cast<int*>(bits + words);
    const int tid = threadIdx.x;
    const double* sc = scores + (long long)blockIdx.x * n;
    for (int w = tid; w < words; w += kLayThreads) bits[w] = 0u;
    for (int w = tid; w < cwords; w += kLayThreads) cand[w] = 0u;
    if (tid == 0) s_chosen = 0;
    const bool chunked = a.layout == 1;
    if (chunked) {
        for (int i = tid; i < N; i += kLayThreads) {
            const int r0 = i * a.B, r1 = min(n, r0 + a.B);
            double s = 0.0;
            for (int j = r0; j < r1; ++j) s += sc[j];  // row by row, in index order
            key[i] = lay_ord(s / (double)(r1 - r0));
        }
    } else {
        for (int i = tid; i < N; i += kLayThreads) key[i] = lay_ord(sc[i]);
    }
    __syncthreads();
    const int m = chunked ? (a.skipped ? 0 : a.c) : min(N, a.k);
    lay_top(key, N, m, cand, hist, warp_sums, &s_prefix, &s_remaining);
    if (a.layout == 0) {
        for (int w = tid; w < words; w += kLayThreads) bits[w] = cand[w];
        if (tid == 0) s_chosen = m;
    } else if (chunked) {
        int mine = 0;
        for (int i = tid; i < N; i += kLayThreads) {
            if (!((cand[i >> 5] >> (i & 31)) & 1u)) continue;
            const int r0 = i * a.B, r1 = min(n, r0 + a.B);
            for (int r = r0; r < r1; ++r) atomicOr(&bits[r >> 5], 1u << (r & 31));
            mine += r1 - r0;
        }
        atomicAdd(&s_chosen, mine);
    } else {
        // the walk never looks past the k best rows in score order (every position it has
        // passed holds a row it has taken, and it stops at k rows): sort those
        const int per = (cwords + kLayThreads - 1) / kLayThreads;
        const int w0 = min(cwords, tid * per), w1 = min(cwords, w0 + per);
        int cnt = 0;
        for (int w = w0; w < w1; ++w) cnt += __popc(cand[w]);
        int tot;
        int pos = lay_scan(cnt, warp_sums, &tot);
        for (int w = w0; w < w1; ++w) {
            uint32_t msk = cand[w];
            while (msk) {
                const int b = __ffs(msk) - 1;
                msk &= msk - 1;
                if (pos < P) order[pos] = w * 32 + b;
                ++pos;
            }
        }
        for (int i = tot + tid; i < P; i += kLayThreads) order[i] = -1;
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int t = tid; t < P / 2; t += kLayThreads) {
                    const int i = (t / stride) * 2 * stride + (t % stride), j = i + stride;
                    const bool up = (i & size) == 0;
                    const int oi = order[i], oj = order[j];
                    if (lay_before(key, oj, oi) == up) {
                        order[i] = oj;
                        order[j] = oi;
                    }
                }
                __syncthreads();
            }
        }
        if (tid == 0) {
            auto marked = [&](int r) { return (bits[r >> 5] >> (r & 31)) & 1u; };
            auto mark = [&](int r) { bits[r >> 5] |= 1u << (r & 31); };
            int chosen = 0, p = 0;
            while (chosen < a.k && p < tot) {
                while (p < tot && marked(order[p])) ++p;
                if (p >= tot) break;
                const int seed = order[p];
                int lo = seed, hi = seed;
                mark(seed);
                ++chosen;
                const unsigned long long thr = lay_ord(a.tau * lay_unord(key[seed]));
                while (chosen < a.k) {
                    const bool l_ok = lo > 0 && !marked(lo - 1) && key[lo - 1] >= thr;
                    const bool r_ok = hi < n - 1 && !marked(hi + 1) && key[hi + 1] >= thr;
                    if (!l_ok && !r_ok) break;
                    if (l_ok && (!r_ok || key[lo - 1] >= key[hi + 1])) mark(--lo);
                    else mark(++hi);
                    ++chosen;
                }
            }
            s_chosen = chosen;
        }
    }
    __syncthreads();
    // ascending row list from the bitmap: each thread owns a run of words
    const int per = (words + kLayThreads - 1) / kLayThreads;
    const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int total;
    int pos = lay_scan(cnt, warp_sums, &total);
    int32_t* out = idx + (long long)blockIdx.x * a.max_rows;
    for (int w = w0; w < w1; ++w) {
        uint32_t msk = bits[w];
        while (msk) {
            const int b = __ffs(msk) - 1;
            msk &= msk - 1;
            if (pos < a.max_rows) out[pos] = w * 32 + b;
            ++pos;
        }
    }
    for (int t = total + tid; t < a.max_rows; t += kLayThreads) out[t] = -1;
    if (tid == 0) {
        counts[blockIdx.x] = total;
        if (total != s_chosen || total > a.max_rows) atomicOr(&g_status_layout, FLAG_BOUNDS);
    }
}

// Keys, the two bitmaps and (grow) the sort buffer of min(N, k) indices padded to a
// power of two.
static int layout_sort_len(int N, int layout, int k) {
    if (layout != 2) return 0;
    const int m = N < k ? N : k;
    int P = 1;
    while (P < m) P <<= 1;
    return P;
}

size_t layout_smem_bytes(int n, int layout, int B, int k) {
    const int N = layout == 1 ? (n + B - 1) / B : n;
    return (size_t)8 * N + (size_t)4 * ((N + 31) / 32) + (size_t)4 * ((n + 31) / 32) +
           (size_t)4 * layout_sort_len(N, layout, k) + 16;
}

cudaError_t launch_repair_layout(const double* scores, int units, int n, int layout, int B, int k, int c,
                                 int skipped, double tau, int32_t* idx, int max_rows, int32_t* counts,
                                 cudaStream_t s) {
    if (units == 0) return cudaSuccess;
    LayoutArgs a;
    a.n = n;
    a.layout = layout;
    a.B = B;
    a.k = k;
    a.c = c;
    a.skipped = skipped;
    a.tau = tau;
    a.max_rows = max_rows;
    const int N = layout == 1 ? (n + B - 1) / B : n;
    const int P = layout_sort_len(N, layout, k);
    const size_t smem = layout_smem_bytes(n, layout, B, k);
    cudaError_t e = cudaFuncSetAttribute(repair_layout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    repair_layout_kernel<<<units, kLayThreads, smem, s>>>(scores, a, N, P, idx, counts);
    return cudaGetLastError();
}

}  // namespace kvfix
