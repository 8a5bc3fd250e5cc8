// diff.cu -- block-sparse sibling diffs against one master cache (kvfix_diff_encode,
// kvfix_diff_gather, kvfix_diff_restore).
//
// Method: TokenDance section 4.3 (master-mirror layout, block-sparse K/V diff) and
// section 5 (touched block indices plus those blocks' K/V contents, one index list
// shared by K and V); section 4.4, Algorithm 1 (restore = master block, overwritten
// where the diff touches it, keys re-aligned by RoPERecover, rows written to a paged
// pool through a slot mapping).
//
// An entry i = (s*L + l)*nblk + blk is bt token rows x all heads x both planes.  Encode
// compares each master block (staged in shared memory by TMA) with every sibling's block
// streaming through a TMA ring; gather holds the master block in registers and writes
// it (or the payload block) for every sibling; restore does the same with the keys
// rotated per sibling and the rows scattered to pool slots.  The master is read once.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

static __device__ unsigned int g_status_diff;

unsigned read_status_diff(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_diff, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_diff, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

constexpr int kDiffThreads = 512;
constexpr int kDiffVec = 8;                             // 16-byte vectors per thread per pass
constexpr int kDiffPass = kDiffThreads * kDiffVec;      // vectors per pass

// Vector q of an entry (K vectors first, then V) -> element offset within the plane.
struct BlockMap {
    int bt, row8;  // tokens per block, vectors per token row
    long long vecs_per_plane;
    __device__ __forceinline__ void locate(long long q, const Plane& p, int c, int l, int t0,
                                           int* plane, long long* off) const {
        *plane = q >= vecs_per_plane;
        long long r = *plane ? q - vecs_per_plane : q;
        int t = (int)(r / row8);
        int c8 = (int)(r % row8);
        *off = p.row(c, l, t0 + t) + 8ll * c8;
    }
};

__device__ __forceinline__ bool vec_ne(const uint4& a, const uint4& b) {
    return ((a.x ^ b.x) | (a.y ^ b.y) | (a.z ^ b.z) | (a.w ^ b.w)) != 0u;
}

// grid = (nblk, L), one CTA per (layer, block).  Sets the mask bits of dirty entries
// (mask pre-zeroed).  The block is cut into "pieces" (a run of rows of one plane, at most
// 32 KB).  The master's piece is bulk-copied (TMA) into one of two master buffers and
// compared with the same piece of every sibling, which stream through a 4-stage ring of
// bulk copies; a sibling's entry is dirty if any piece differs.  The master is read once.
// Warp 15 (one lane) issues the copies; warps 0..14 compare.  A comparing warp ORs its
// verdict into the sibling's flag and releases the stage (and, after a piece's last
// sibling, the master buffer) by an arrive on an "empty" mbarrier, so the warps never
// wait for one another between pieces.
constexpr int kDmThreads = 512;
constexpr int kDmCmpWarps = kDmThreads / 32 - 1;  // comparing warps
constexpr int kDmStages = 4;
constexpr int kDmPieceBytes = 32768;

struct DmArgs {
    const uint16_t* mk;
    const uint16_t* mv;
    const uint16_t* sk;
    const uint16_t* sv;
    Plane mp, sp;
    int bt, piece_rows, pieces_per_plane;
    uint32_t* mask;    // K and V together, or K alone when mask_v is set
    uint32_t* mask_v;  // V alone (per-plane lists), or null
};

__global__ void __launch_bounds__(kDmThreads, 1) diff_mask_kernel(DmArgs a) {
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t mfull[2], mempty[2], full[kDmStages], empty[kDmStages];
    __shared__ int abort_flag;
    const int blk = blockIdx.x, l = blockIdx.y;
    const int S = a.sp.chunks, L = a.mp.layers, nblk = a.mp.tokens / a.bt;
    const int HD = a.mp.heads * a.mp.dim;
    const unsigned row_bytes = (unsigned)HD * 2u;
    const int P = 2 * a.pieces_per_plane;  // pieces per block (K pieces, then V pieces)
    const int units = P * S;               // (piece, sibling) pairs, piece-major
    unsigned char* mbuf = dsm;                                 // [2][kDmPieceBytes]
    unsigned char* ring = dsm + 2 * kDmPieceBytes;             // [kDmStages][kDmPieceBytes]
    uint32_t* flags = reinterpret_cast<uint32_t*>(ring + kDmStages * kDmPieceBytes);  // [planes][ceil(S/32)]
    const int fwords = (S + 31) / 32;
    const bool split = a.mask_v != nullptr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool contig_m = a.mp.st == HD, contig_s = a.sp.st == HD;

    // piece p: plane p / pieces_per_plane, rows [r0, r0 + rows) of the block
    auto piece_rows = [&](int p, int* r0) {
        const int q = p % a.pieces_per_plane;
        *r0 = q * a.piece_rows;
        return min(a.piece_rows, a.bt - *r0);
    };
    auto copy_rows = [&](unsigned char* dst, const uint16_t* base, const Plane& pl, int chunk, int t0, int rows,
                         bool contig, uint64_t* bar) {
        if (contig) {
            bulk_g2s(dst, base + pl.row(chunk, l, t0), row_bytes * rows, bar);
        } else {
            for (int q = 0; q < rows; ++q) bulk_g2s(dst + q * row_bytes, base + pl.row(chunk, l, t0 + q), row_bytes, bar);
        }
    };

    for (int i = tid; i < (split ? 2 : 1) * fwords; i += kDmThreads) flags[i] = 0u;
    if (tid == 0) {
        for (int q = 0; q < 2; ++q) {
            mbar_init(&mfull[q], 1);
            mbar_init(&mempty[q], kDmCmpWarps);
        }
        for (int q = 0; q < kDmStages; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], kDmCmpWarps);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();

    if (warp == kDmCmpWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int g = 0; g < units; ++g) {
                const int p = g / S, s = g % S;
                int r0;
                const int rows = piece_rows(p, &r0);
                const bool vpl = p >= a.pieces_per_plane;
                if (s == 0) {  // the piece's master, once its buffer's previous piece is done
                    if (p >= 2 && !mbar_wait(&mempty[p & 1], (unsigned)((p >> 1) - 1) & 1u)) {
                        atomicOr(&abort_flag, 1);
                        break;
                    }
                    mbar_arrive_expect_tx(&mfull[p & 1], row_bytes * rows);
                    copy_rows(mbuf + (p & 1) * kDmPieceBytes, vpl ? a.mv : a.mk, a.mp, 0, blk * a.bt + r0, rows,
                              contig_m, &mfull[p & 1]);
                }
                const int slot = g % kDmStages;
                if (g >= kDmStages && !mbar_wait(&empty[slot], (unsigned)(g / kDmStages - 1) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                mbar_arrive_expect_tx(&full[slot], row_bytes * rows);
                copy_rows(ring + slot * kDmPieceBytes, vpl ? a.sv : a.sk, a.sp, s, blk * a.bt + r0, rows, contig_s,
                          &full[slot]);
            }
        }
    } else {
        // ------------------------------------------------------------ compare
        const int ct = tid;  // 0 .. 32*kDmCmpWarps - 1
        for (int g = 0; g < units; ++g) {
            const int p = g / S, s = g % S;
            int r0;
            const int rows = piece_rows(p, &r0);
            bool ok = !abort_flag;
            if (ok && s == 0) ok = mbar_wait(&mfull[p & 1], (unsigned)(p >> 1) & 1u);
            ok = ok && mbar_wait(&full[g % kDmStages], (unsigned)(g / kDmStages) & 1u);
            if (!ok) {
                atomicOr(&abort_flag, 1);
                break;
            }
            const uint4* m4 = reinterpret_cast<const uint4*>(mbuf + (p & 1) * kDmPieceBytes);
            const uint4* s4 = reinterpret_cast<const uint4*>(ring + (g % kDmStages) * kDmPieceBytes);
            const int vecs = rows * (int)(row_bytes / 16);
            bool ne = false;
            for (int v = ct; v < vecs; v += 32 * kDmCmpWarps) ne |= vec_ne(m4[v], s4[v]);
            const int fp = split && p >= a.pieces_per_plane ? fwords : 0;  // the V plane's flags
            if (__any_sync(0xffffffffu, ne) && lane == 0) atomicOr(&flags[fp + (s >> 5)], 1u << (s & 31));
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[g % kDmStages]);
                if (s == S - 1) mbar_arrive(&mempty[p & 1]);
            }
        }
    }
    __syncthreads();
    if (abort_flag) {
        if (tid == 0) {
            atomicOr(&g_status_diff, FLAG_TIMEOUT);
            // copies possibly in flight: wait (bounded) on both phases of every barrier
            for (int q = 0; q < 2; ++q) mbar_wait(&mfull[q], 0u), mbar_wait(&mfull[q], 1u);
            for (int q = 0; q < kDmStages; ++q) mbar_wait(&full[q], 0u), mbar_wait(&full[q], 1u);
        }
        __syncthreads();
        return;
    }
    for (int q = tid; q < (split ? 2 : 1) * S; q += kDmThreads) {
        const int pl = q / S, sq = q % S;
        if (flags[pl * fwords + (sq >> 5)] >> (sq & 31) & 1u) {
            const long long i = ((long long)sq * L + l) * nblk + blk;
            atomicOr(&(pl ? a.mask_v : a.mask)[i >> 5], 1u << (i & 31));
        }
    }
}

cudaError_t launch_diff_mask(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                             const uint16_t* sk, const uint16_t* sv, const kvfix_kv_desc& sd,
                             int bt, uint32_t* mask, cudaStream_t s, uint32_t* mask_v) {
    DmArgs a;
    a.mk = mk;
    a.mv = mv;
    a.sk = sk;
    a.sv = sv;
    a.mp = plane_of(md);
    a.sp = plane_of(sd);
    a.bt = bt;
    a.mask = mask;
    a.mask_v = mask_v;
    if (a.mp.layers == 0 || a.mp.tokens == 0 || a.sp.chunks == 0) return cudaSuccess;
    const int row_bytes = 2 * a.mp.heads * a.mp.dim;
    a.piece_rows = kDmPieceBytes / row_bytes < bt ? kDmPieceBytes / row_bytes : bt;
    if (a.piece_rows < 1) return cudaErrorInvalidValue;  // a token row above 32 KB
    a.pieces_per_plane = (bt + a.piece_rows - 1) / a.piece_rows;
    const size_t smem = (size_t)(2 + kDmStages) * kDmPieceBytes + 8 * (size_t)((a.sp.chunks + 31) / 32);
    cudaError_t e = cudaFuncSetAttribute(diff_mask_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.mp.tokens / bt, a.mp.layers);
    diff_mask_kernel<<<grid, kDmThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------- scan
constexpr int kScanThreads = 1024;

__device__ __forceinline__ int mask_bit(const uint32_t* mask, long long i) {
    return (mask[i >> 5] >> (i & 31)) & 1;
}

// Exclusive scan of one value per thread (long long), block total in *total.
__device__ long long block_scan_ll(long long x, long long* ws, long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) ws[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        long long v = lane < nw ? ws[lane] : 0, vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, vi, o);
            if (lane >= o) vi += y;
        }
        if (lane < nw) ws[lane] = vi - v;
        if (lane == 31) ws[32] = vi;
    }
    __syncthreads();
    long long ex = inc - x + ws[warp];
    *total = ws[32];
    __syncthreads();
    return ex;
}

// grid = siblings.  offsets[s*P + k] = dirty entries before it (over all siblings).
__global__ void __launch_bounds__(kScanThreads)
diff_scan_kernel(const uint32_t* __restrict__ mask, long long P, int S, int64_t* offsets) {
    __shared__ long long ws[33];
    const int s = blockIdx.x;
    const long long lo = (long long)s * P;  // first entry of this sibling
    // dirty entries of earlier siblings: bits [0, lo)
    long long before = 0;
    const long long full_words = lo >> 5;
    for (long long w = threadIdx.x; w < full_words; w += blockDim.x) before += __popc(mask[w]);
    if (threadIdx.x == 0 && (lo & 31)) before += __popc(mask[full_words] & ((1u << (lo & 31)) - 1u));
    long long tot;
    block_scan_ll(before, ws, &tot);
    const long long base = tot;
    const long long seg = (P + blockDim.x - 1) / blockDim.x;
    const long long i0 = min(P, (long long)threadIdx.x * seg), i1 = min(P, i0 + seg);
    long long cnt = 0;
    for (long long i = i0; i < i1; ++i) cnt += mask_bit(mask, lo + i);
    long long run = base + block_scan_ll(cnt, ws, &tot);
    for (long long i = i0; i < i1; ++i) {
        offsets[lo + i] = run;
        run += mask_bit(mask, lo + i);
    }
    if (s == S - 1 && threadIdx.x == 0) offsets[(long long)S * P] = base + tot;
}

cudaError_t launch_diff_scan(const uint32_t* mask, int siblings, long long per_sibling,
                             int64_t* offsets, cudaStream_t s) {
    if (siblings == 0) return cudaMemsetAsync(offsets, 0, sizeof(int64_t), s);
    diff_scan_kernel<<<siblings, kScanThreads, 0, s>>>(mask, per_sibling, siblings, offsets);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------- pack
constexpr int kPackThreads = 256;

// grid = ceil(E/32): one CTA per mask word; copies each dirty entry to the payload.
__global__ void __launch_bounds__(kPackThreads)
diff_pack_kernel(const uint16_t* __restrict__ sk, const uint16_t* __restrict__ sv, Plane sp, int bt,
                 const uint32_t* __restrict__ mask, const int64_t* __restrict__ offsets,
                 long long E, uint16_t* payload, long long capacity, int planes) {
    const long long wi = blockIdx.x;
    uint32_t word = mask[wi];
    const int L = sp.layers, nblk = sp.tokens / bt;
    BlockMap bm{bt, sp.heads * sp.dim / 8, (long long)bt * (sp.heads * sp.dim / 8)};
    // planes: 0 = the block's K rows then its V rows, 1 = K rows only, 2 = V rows only
    const long long total = (planes == 0 ? 2 : 1) * bm.vecs_per_plane;
    const long long vbase = planes == 2 ? bm.vecs_per_plane : 0;
    while (word) {
        const int bit = __ffs(word) - 1;
        word &= word - 1;
        const long long i = wi * 32 + bit;
        if (i >= E) break;
        const long long e = offsets[i];
        if (e >= capacity) {
            if (threadIdx.x == 0) atomicOr(&g_status_diff, FLAG_NOSPACE);
            continue;
        }
        const int s = (int)(i / ((long long)L * nblk));
        const int l = (int)((i / nblk) % L);
        const int blk = (int)(i % nblk);
        uint4* dst = reinterpret_cast<uint4*>(payload + e * total * 8);
        const int row8 = bm.row8, rows_all = (planes == 0 ? 2 : 1) * bt;
        const int rshift = planes == 2 ? bt : 0;  // first source row, counted over K then V
        if (kPackThreads % row8 == 0) {
            // a thread keeps one 16-byte column and walks rows; eight loads in flight
            const int rpp = kPackThreads / row8, c8 = threadIdx.x % row8, r0 = threadIdx.x / row8;
            const long long boff = sp.row(s, l, blk * bt) + 8 * c8;
            for (int rb = 0; rb < rows_all; rb += 8 * rpp) {
                uint4 v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int r = rb + r0 + j * rpp, rr = r + rshift;
                    if (r < rows_all)
                        v[j] = ld_stream(reinterpret_cast<const uint4*>(
                            (rr < bt ? sk + boff + (long long)rr * sp.st : sv + boff + (long long)(rr - bt) * sp.st)));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int r = rb + r0 + j * rpp;
                    if (r < rows_all) st_stream(dst + (long long)r * row8 + c8, v[j]);
                }
            }
        } else {
            for (long long q = threadIdx.x; q < total; q += kPackThreads) {
                int pl;
                long long off;
                bm.locate(q + vbase, sp, s, l, blk * bt, &pl, &off);
                uint4 v = ld_stream(reinterpret_cast<const uint4*>((pl ? sv : sk) + off));
                st_stream(dst + q, v);
            }
        }
    }
}

cudaError_t launch_diff_pack(const uint16_t* sk, const uint16_t* sv, const kvfix_kv_desc& sd,
                             int bt, const uint32_t* mask, const int64_t* offsets,
                             uint16_t* payload, long long capacity, cudaStream_t s, int planes) {
    Plane sp = plane_of(sd);
    const long long E = (long long)sp.chunks * sp.layers * (sp.tokens / bt);
    if (E == 0) return cudaSuccess;
    const long long words = (E + 31) / 32;
    diff_pack_kernel<<<(unsigned)words, kPackThreads, 0, s>>>(sk, sv, sp, bt, mask, offsets, E,
                                                              payload, capacity, planes);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------- gather

constexpr int kGatherSibChunk = 64;  // siblings whose payload entries a CTA stages at once

// The V plane's list when K and V keep separate ones (null mask: one list for both).
struct SplitList {
    const uint32_t* mask;
    const int64_t* offsets;
    const uint16_t* payload;
    long long entries;
};

// Payload entry of sibling entry i in a list, or -1 (clean, or beyond the payload: flagged).
__device__ __forceinline__ long long diff_entry(const uint32_t* mask, const int64_t* offsets, long long entries,
                                               long long i) {
    long long e = mask_bit(mask, i) ? offsets[i] : -1;
    if (e >= entries) {
        atomicOr(&g_status_diff, FLAG_NOSPACE);
        e = -1;
    }
    return e;
}

// grid = (nblk, L).  Master block in registers, written to every sibling unless the
// sibling's entry is dirty, in which case the payload block is copied instead.  With a
// split list, K blocks come from (mask, offsets, payload) and V blocks from vl, each
// payload entry holding one plane.
__global__ void __launch_bounds__(kDiffThreads)
diff_gather_kernel(const uint16_t* __restrict__ mk, const uint16_t* __restrict__ mv, Plane mp,
                   const uint32_t* __restrict__ mask, const int64_t* __restrict__ offsets,
                   const uint16_t* __restrict__ payload, long long payload_entries, int S, int bt,
                   uint16_t* ok, uint16_t* ov, Plane op, SplitList vl) {
    __shared__ long long ent_k[kGatherSibChunk], ent_v[kGatherSibChunk];
    const int blk = blockIdx.x, l = blockIdx.y;
    const int nblk = mp.tokens / bt, L = mp.layers;
    BlockMap bm{bt, mp.heads * mp.dim / 8, (long long)bt * (mp.heads * mp.dim / 8)};
    const long long total = 2 * bm.vecs_per_plane;
    for (long long q0 = 0; q0 < total; q0 += kDiffPass) {
        uint4 m[kDiffVec];
        int pl[kDiffVec];
        long long off[kDiffVec];
#pragma unroll
        for (int k = 0; k < kDiffVec; ++k) {
            long long q = q0 + (long long)k * kDiffThreads + threadIdx.x;
            pl[k] = -1;
            if (q < total) {
                long long o;
                bm.locate(q, mp, 0, l, blk * bt, &pl[k], &o);
                m[k] = *reinterpret_cast<const uint4*>((pl[k] ? mv : mk) + o);
                bm.locate(q, op, 0, l, blk * bt, &pl[k], &off[k]);
            }
        }
        const bool split = vl.mask != nullptr;
        const long long vpp = bm.vecs_per_plane, estride = split ? vpp : total;
        // the payload entries of a chunk of siblings, looked up once per CTA
        for (int s0 = 0; s0 < S; s0 += kGatherSibChunk) {
            const int sc = min(kGatherSibChunk, S - s0);
            __syncthreads();  // the previous chunk's entries are no longer read
            if (threadIdx.x < sc) {
                const long long i = ((long long)(s0 + threadIdx.x) * L + l) * nblk + blk;
                ent_k[threadIdx.x] = diff_entry(mask, offsets, payload_entries, i);
                ent_v[threadIdx.x] = split ? diff_entry(vl.mask, vl.offsets, vl.entries, i) : -1;
            }
            __syncthreads();
            for (int ss = 0; ss < sc; ++ss) {
                const int s = s0 + ss;
                const long long e = ent_k[ss];
                const uint4* src = e >= 0 ? reinterpret_cast<const uint4*>(payload + e * estride * 8) : nullptr;
                const uint4* srcv = src;  // joint entry: V vectors follow its K vectors
                if (split) {
                    const long long ev = ent_v[ss];
                    srcv = ev >= 0 ? reinterpret_cast<const uint4*>(vl.payload + ev * vpp * 8) : nullptr;
                }
#pragma unroll
                for (int k = 0; k < kDiffVec; ++k) {
                    if (pl[k] < 0) continue;
                    const long long q = q0 + (long long)k * kDiffThreads + threadIdx.x;
                    const uint4* sp = pl[k] ? srcv : src;
                    uint4 v = sp ? ld_stream(sp + (split && pl[k] ? q - vpp : q)) : m[k];
                    uint16_t* base = (pl[k] ? ov : ok) + (long long)s * op.sc;
                    st_stream(reinterpret_cast<uint4*>(base + off[k]), v);
                }
            }
        }
    }
}

cudaError_t launch_diff_gather(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                               const uint32_t* mask, const int64_t* offsets,
                               const uint16_t* payload, long long payload_entries, int siblings,
                               int bt, uint16_t* ok, uint16_t* ov, const kvfix_kv_desc& od,
                               cudaStream_t s, const uint32_t* mask_v, const int64_t* offsets_v,
                               const uint16_t* payload_v, long long entries_v) {
    Plane mp = plane_of(md), op = plane_of(od);
    if (mp.layers == 0 || mp.tokens == 0 || siblings == 0) return cudaSuccess;
    dim3 grid(mp.tokens / bt, mp.layers);
    SplitList vl{mask_v, offsets_v, payload_v, entries_v};
    diff_gather_kernel<<<grid, kDiffThreads, 0, s>>>(mk, mv, mp, mask, offsets, payload,
                                                     payload_entries, siblings, bt, ok, ov, op, vl);
    return cudaGetLastError();
}

// --------------------------------------------------------------- master selection

constexpr int kMsThreads = 256;

// grid = agents.  total[a] = sum over the agent's units and tokens of d_k + d_v, in double:
// thread t takes every 256th value of the agent's range, then a fixed tree over threads.
__global__ void __launch_bounds__(kMsThreads)
master_total_kernel(const float* __restrict__ d_k, const float* __restrict__ d_v, long long per_agent,
                    double* totals) {
    __shared__ double part[kMsThreads];
    const long long base = (long long)blockIdx.x * per_agent;
    double s = 0.0;
    for (long long i = threadIdx.x; i < per_agent; i += kMsThreads) {
        if (d_k) s += (double)d_k[base + i];
        if (d_v) s += (double)d_v[base + i];
    }
    part[threadIdx.x] = s;
    __syncthreads();
    for (int h = kMsThreads / 2; h > 0; h >>= 1) {
        if (threadIdx.x < h) part[threadIdx.x] += part[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = part[0];
}

// One warp: the smallest total, ties to the lower agent.
__global__ void master_argmin_kernel(const double* __restrict__ totals, int A, int32_t* master) {
    double best = 0.0;
    int bi = -1;
    for (int a = threadIdx.x; a < A; a += 32)
        if (bi < 0 || totals[a] < best) {
            best = totals[a];
            bi = a;
        }
    for (int o = 16; o > 0; o >>= 1) {
        const double ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi >= 0 && (bi < 0 || ob < best || (ob == best && oi < bi))) {
            best = ob;
            bi = oi;
        }
    }
    if (threadIdx.x == 0) *master = bi;
}

cudaError_t launch_master_select(const float* d_k, const float* d_v, int agents, int units_per_agent,
                                 int tokens, double* totals, int32_t* master, cudaStream_t s) {
    if (agents == 0) return cudaSuccess;
    master_total_kernel<<<agents, kMsThreads, 0, s>>>(d_k, d_v, (long long)units_per_agent * tokens, totals);
    master_argmin_kernel<<<1, 32, 0, s>>>(totals, agents, master);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------- restore

constexpr int kRestoreThreads = 512;
constexpr int kRestoreSibChunk = 16;                 // siblings per staged chunk
constexpr int kRestoreSlotStage = 4096;              // staged (sibling, token) slots

// Rotate (x_i, x_{i+D/2}) for the 8 dims of one pair item: (lo, hi) bf16 vectors; c, s,
// m hold (cos, sin, -sin) of the 8 angles as float pairs.  Per element the same operations,
// and so the same rounding, as kvfix_rerope (fma(x0, c, x1 * -s), fma(x1, c, x0 * s)), two
// lanes at a time.
__device__ __forceinline__ void restore_rotate8(uint4& lo, uint4& hi, const float2* c,
                                                const float2* s, const float2* m) {
    __nv_bfloat162* l2 = reinterpret_cast<__nv_bfloat162*>(&lo);
    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&hi);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 x0 = __bfloat1622float2(l2[q]), x1 = __bfloat1622float2(h2[q]);
        l2[q] = __float22bfloat162_rn(__ffma2_rn(x0, c[q], __fmul2_rn(x1, m[q])));
        h2[q] = __float22bfloat162_rn(__ffma2_rn(x1, c[q], __fmul2_rn(x0, s[q])));
    }
}

// grid = (nblk, L).  A thread owns one pair column r of the token row (the 8-wide K
// vectors at dims 8j and D/2 + 8j of one head, which rotate together, j = r mod D/16) and
// two V vector columns, for two rows of the block at a time; the master's pieces stay in
// registers while every sibling is written.  Since the column is fixed, the sibling's
// (cos, sin, -sin) of the column's 8 angles are read once for both rows.  Siblings go in
// chunks of up to 16: per chunk the CTA stages in shared memory each sibling's payload
// entry (or -1), its angle tables and the pool slots of the pass's rows, so the
// per-sibling loop issues its stores without waiting on global memory.  With per-plane
// lists (vl.mask set) each sibling has a K entry in the first list and a V entry in vl,
// each holding one plane's block.
__global__ void __launch_bounds__(kRestoreThreads, 1)
diff_restore_kernel(const uint16_t* __restrict__ mk, const uint16_t* __restrict__ mv, Plane mp,
                    const uint32_t* __restrict__ mask, const int64_t* __restrict__ offsets,
                    const uint16_t* __restrict__ payload, long long payload_entries, int S, int bt,
                    const int32_t* __restrict__ delta, RopeTheta th,
                    const int32_t* __restrict__ slot_map, uint16_t* pk, uint16_t* pv, Plane pp, SplitList vl) {
    __shared__ __align__(16) float cos_s[kRestoreSibChunk][kMaxHeadDim / 2];
    __shared__ __align__(16) float sin_s[kRestoreSibChunk][kMaxHeadDim / 2];
    __shared__ __align__(16) float nsin_s[kRestoreSibChunk][kMaxHeadDim / 2];
    __shared__ int slot_s[kRestoreSlotStage];
    __shared__ long long ent_s[kRestoreSibChunk], entv_s[kRestoreSibChunk];
    const bool split = vl.mask != nullptr;  // per-plane lists: each payload entry holds one plane
    __shared__ int rot_s[kRestoreSibChunk];
    const int blk = blockIdx.x, l = blockIdx.y;
    const int n = mp.tokens, nblk = n / bt, L = mp.layers;
    const int D = mp.dim, half = D / 2, hp = D / 16;
    const int rowe = mp.heads * D;                           // elements per token row
    const int P = rowe / 16;                                 // pair columns per row
    const int Pc = min(P, kRestoreThreads);                  // pair columns per segment
    const int rpp = kRestoreThreads / Pc;                    // row slots per segment
    const int rc = threadIdx.x % Pc, trow = threadIdx.x / Pc;
    const bool active = trow < rpp;
    const long long blk_elems = (long long)bt * rowe;        // elements per plane of a block
    const int t0 = blk * bt;
    const int slots = pp.tokens;
    uint16_t* pkl = pk + (long long)l * pp.sl;
    uint16_t* pvl = pv + (long long)l * pp.sl;
    for (int c0 = 0; c0 < P; c0 += Pc) {
        const int r = c0 + rc;
        const bool k_ok = active && r < P;
        const int ki = 8 * (r % hp), ke = (r / hp) * D + ki;   // angle index, element offset
        int vo[2];
        bool v_ok[2];
        vo[0] = 8 * (2 * c0 + rc);
        vo[1] = vo[0] + 8 * Pc;
        v_ok[0] = active && vo[0] < rowe;
        v_ok[1] = active && vo[1] < rowe;
        for (int row0 = 0; row0 < bt; row0 += 2 * rpp) {
            const int tpn = min(2 * rpp, bt - row0);
            const int chunk = max(1, min(kRestoreSibChunk, kRestoreSlotStage / tpn));
            int row[2];
            row[0] = trow;            // rows of the pass, relative to row0
            row[1] = trow + rpp;
            uint4 klo[2], khi[2], vv[2][2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (!active || row[x] >= tpn) {
                    row[x] = -1;
                    continue;
                }
                const long long base = mp.row(0, l, t0 + row0 + row[x]);
                if (k_ok) {
                    klo[x] = ld_stream(reinterpret_cast<const uint4*>(mk + base + ke));
                    khi[x] = ld_stream(reinterpret_cast<const uint4*>(mk + base + ke + half));
                }
#pragma unroll
                for (int y = 0; y < 2; ++y)
                    if (v_ok[y]) vv[x][y] = ld_stream(reinterpret_cast<const uint4*>(mv + base + vo[y]));
            }
            for (int s0 = 0; s0 < S; s0 += chunk) {
                const int sc = min(chunk, S - s0);
                __syncthreads();  // the previous chunk's stage is no longer read
                for (int x = threadIdx.x; x < sc * half; x += kRestoreThreads) {
                    const int ss = x / half, i = x % half;
                    float c, sn;
                    rope_cos_sin(delta[s0 + ss], th.theta[i], &c, &sn);
                    cos_s[ss][i] = c;
                    sin_s[ss][i] = sn;
                    nsin_s[ss][i] = -sn;
                }
                for (int x = threadIdx.x; x < sc * tpn; x += kRestoreThreads) {
                    const int ss = x / tpn, tt = x % tpn;
                    int slot = __ldg(slot_map + (long long)(s0 + ss) * n + t0 + row0 + tt);
                    if (slot >= slots) {
                        atomicOr(&g_status_diff, FLAG_BOUNDS);
                        slot = -1;
                    }
                    slot_s[x] = slot;
                }
                if (threadIdx.x < sc) {
                    const int s = s0 + threadIdx.x;
                    const long long i = ((long long)s * L + l) * nblk + blk;
                    ent_s[threadIdx.x] = diff_entry(mask, offsets, payload_entries, i);
                    entv_s[threadIdx.x] = split ? diff_entry(vl.mask, vl.offsets, vl.entries, i) : -1;
                    rot_s[threadIdx.x] = delta[s] != 0;
                }
                __syncthreads();
                for (int ss = 0; ss < sc; ++ss) {
                    const long long e = ent_s[ss];
                    const uint16_t* src = e >= 0 ? payload + e * (split ? 1 : 2) * blk_elems : nullptr;
                    const uint16_t* srcv;  // the V block: after the K block, or its own list's entry
                    if (split) {
                        const long long ev = entv_s[ss];
                        srcv = ev >= 0 ? vl.payload + ev * blk_elems : nullptr;
                    } else {
                        srcv = src ? src + blk_elems : nullptr;
                    }
                    const bool rotate = rot_s[ss] != 0 && k_ok;
                    float2 cc[4], sn[4], ns[4];
                    if (rotate) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            cc[q] = reinterpret_cast<const float2*>(&cos_s[ss][ki])[q];
                            sn[q] = reinterpret_cast<const float2*>(&sin_s[ss][ki])[q];
                            ns[q] = reinterpret_cast<const float2*>(&nsin_s[ss][ki])[q];
                        }
                    }
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (row[x] < 0) continue;
                        const int slot = slot_s[ss * tpn + row[x]];
                        if (slot < 0) continue;
                        const long long prow = (long long)slot * pp.st;
                        const long long srow = (long long)(row0 + row[x]) * rowe;
                        if (k_ok) {
                            uint4 a = klo[x], b = khi[x];
                            if (src) {
                                a = ld_stream(reinterpret_cast<const uint4*>(src + srow + ke));
                                b = ld_stream(reinterpret_cast<const uint4*>(src + srow + ke + half));
                            }
                            if (rotate) restore_rotate8(a, b, cc, sn, ns);
                            st_stream(reinterpret_cast<uint4*>(pkl + prow + ke), a);
                            st_stream(reinterpret_cast<uint4*>(pkl + prow + ke + half), b);
                        }
#pragma unroll
                        for (int y = 0; y < 2; ++y) {
                            if (!v_ok[y]) continue;
                            uint4 v = vv[x][y];
                            if (srcv) v = ld_stream(reinterpret_cast<const uint4*>(srcv + srow + vo[y]));
                            st_stream(reinterpret_cast<uint4*>(pvl + prow + vo[y]), v);
                        }
                    }
                }
            }
        }
    }
}

cudaError_t launch_diff_restore(const uint16_t* mk, const uint16_t* mv, const kvfix_kv_desc& md,
                                const uint32_t* mask, const int64_t* offsets,
                                const uint16_t* payload, long long payload_entries, int siblings,
                                int bt, const int32_t* delta, const RopeTheta& th,
                                const int32_t* slot_map, uint16_t* pk, uint16_t* pv,
                                const kvfix_kv_desc& pd, cudaStream_t s, const uint32_t* mask_v,
                                const int64_t* offsets_v, const uint16_t* payload_v, long long entries_v) {
    Plane mp = plane_of(md), pp = plane_of(pd);
    SplitList vl{mask_v, offsets_v, payload_v, entries_v};
    if (mp.layers == 0 || mp.tokens == 0 || siblings == 0) return cudaSuccess;
    dim3 grid(mp.tokens / bt, mp.layers);
    diff_restore_kernel<<<grid, kRestoreThreads, 0, s>>>(mk, mv, mp, mask, offsets, payload,
                                                         payload_entries, siblings, bt, delta, th,
                                                         slot_map, pk, pv, pp, vl);
    return cudaGetLastError();
}

}  // namespace kvfix
