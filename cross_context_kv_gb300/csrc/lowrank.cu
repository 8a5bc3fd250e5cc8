// lowrank.cu -- kvfix_lowrank_apply: out = x + A B per (chunk, layer, KV head).
//
// Method: KVCMAS Eq. 4 (corrected cache = reference + estimated delta), Eq. 7 (a delta
// kept as factors A [rows x r] and B [r x D]), Eq. 8 with a single anchor of weight 1.
//
// Blackwell path: one CTA per (unit = chunk, layer, head; range of 128-row tiles).
//   warp 0      TMA producer: x tile (128 rows x D, two 64-column boxes, 128-byte
//               swizzle) and A tile (128 rows x r, r*2-byte swizzle) into a ring of up to 5 stages;
//   warp 1      allocates tensor memory and issues tcgen05.mma: one M=128 x N=D x K=16
//               MMA per 16 ranks, float accumulator in TMEM (two buffers);
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows, + x (read from the same
//               stage, swizzled), one rounding to bf16 written back in place, TMA store.
// B of the unit is transposed once into the K-major canonical layout by all threads.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "tc.cuh"

namespace kvfix {

static __device__ unsigned int g_status_lowrank;

unsigned read_status_lowrank(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_lowrank, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_lowrank, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

constexpr int kLtThreads = 192;  // warp 0 producer, warp 1 MMA, warps 2..5 epilogue
constexpr int kLtMaxStages = 5;  // ring depth, as far as shared memory allows
constexpr int kLtSmemLimit = 227 * 1024;
constexpr int kLtRows = 128;     // rows per tile (MMA M)
constexpr int kLtTilesPerCta = 64;

template <int D, int RANK>
struct LtCfg {
    static constexpr int kXBytes = kLtRows * D * 2;            // x tile
    static constexpr int kABytes = kLtRows * RANK * 2;         // A tile
    static constexpr int kStage = ((kXBytes + kABytes) + 1023) / 1024 * 1024;
    static constexpr int kBBytes = D * RANK * 2;
    // as many stages (up to kLtMaxStages) as fit: the ring is what keeps bytes in flight
    static constexpr int kFit = (kLtSmemLimit - 1024 - kBBytes) / kStage;
    static constexpr int kStages = kFit < kLtMaxStages ? kFit : kLtMaxStages;
    static constexpr int kSmem = 1024 /*alignment slack*/ + kStages * kStage + kBBytes;
    static constexpr int kCols = 2 * D;                        // two accumulators (power of 2)
    static constexpr int kASwizzleBytes = RANK * 2;            // 32, 64 or 128
    static constexpr uint32_t kALayout = RANK == 16 ? 6u : RANK == 32 ? 4u : 2u;
};

struct LtArgs {
    const uint16_t* B;  // [units][RANK][D]
    int H, L, n, tiles_per_unit, tiles_per_cta;
};

template <int D, int RANK>
__global__ void __launch_bounds__(kLtThreads, 1)
lowrank_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_out,
                  const __grid_constant__ CUtensorMap tm_a, LtArgs args) {
    using C = LtCfg<D, RANK>;
    extern __shared__ unsigned char smem_raw[];
    constexpr int kLtStages = C::kStages;
    __shared__ __align__(8) uint64_t full[kLtStages], empty[kLtStages], tfull[2], tempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* bsm = smem + kLtStages * C::kStage;  // B, K-major canonical, no swizzle
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, cl = blockIdx.z;
    const int c = cl / args.L, l = cl % args.L;
    const long long unit = (long long)cl * args.H + h;
    const int tile0 = blockIdx.x * args.tiles_per_cta;
    const int ntiles = min(args.tiles_per_cta, args.tiles_per_unit - tile0);

    // B of this unit -> element (e, k) at (e%8)*16 + (e/8)*SBO + (k/8)*128 + (k%8)*2,
    // SBO = (RANK/8)*128: the K-major, unswizzled core-matrix layout.
    const uint16_t* Bu = args.B + unit * (long long)RANK * D;
    for (int i = threadIdx.x; i < RANK * D; i += kLtThreads) {
        const int k = i / D, e = i % D;
        const int off = (e % 8) * 16 + (e / 8) * (RANK / 8) * 128 + (k / 8) * 128 + (k % 8) * 2;
        *reinterpret_cast<uint16_t*>(bsm + off) = Bu[i];
    }
    fence_proxy_async_smem();  // generic writes of B -> read by the tensor core (async proxy)
    if (threadIdx.x == 0) {
        for (int s = 0; s < kLtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        fence_mbar_init();
        abort_flag = 0;
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_out);
        prefetch_tensormap(&tm_a);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, C::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < ntiles && !vload(&abort_flag); ++i) {
                const int s = i % kLtStages;
                if (i >= kLtStages && !mbar_wait(&empty[s], (unsigned)(i / kLtStages - 1) & 1u)) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                unsigned char* st = smem + s * C::kStage;
                const int t0 = (tile0 + i) * kLtRows;
                mbar_arrive_expect_tx(&full[s], C::kXBytes + C::kABytes);
                for (int half = 0; half < D / 64; ++half)
                    tma_load_4d(st + half * (kLtRows * 128), &tm_x, h * D + 64 * half, t0, l, c, &full[s]);
                tma_load_2d(st + C::kXBytes, &tm_a, 0, (int)(unit * args.n + t0), &full[s]);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc_bf16(kLtRows, D);
            for (int i = 0; i < ntiles && !vload(&abort_flag); ++i) {
                const int s = i % kLtStages, a = i & 1;
                if (!mbar_wait(&full[s], (unsigned)(i / kLtStages) & 1u) ||
                    (i >= 2 && !mbar_wait(&tempty[a], (unsigned)(i / 2 - 1) & 1u))) {
                    atomicOr(&abort_flag, 1);
                    break;
                }
                tc_fence_after();
                const unsigned char* at = smem + s * C::kStage + C::kXBytes;
#pragma unroll
                for (int kk = 0; kk < RANK / 16; ++kk) {
                    const uint64_t adesc = tc_smem_desc(at + 32 * kk, 16, 8 * C::kASwizzleBytes, C::kALayout);
                    const uint64_t bdesc = tc_smem_desc(bsm + 256 * kk, 128, (RANK / 8) * 128, 0);
                    tc_mma_bf16(tmem + a * D, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(&tfull[a]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int wq = warp & 3;              // TMEM lane quarter this warp may read
        const int m = 32 * wq + lane;         // tile row of this thread
        const int et = threadIdx.x - 64;      // 0..127
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % kLtStages, a = i & 1;
            bool ok = !vload(&abort_flag) && mbar_wait(&tfull[a], (unsigned)(i / 2) & 1u);
            if (!ok) atomicOr(&abort_flag, 1);
            tc_fence_after();
            unsigned char* st = smem + s * C::kStage;
            if (ok) {
#pragma unroll
                for (int j = 0; j < D / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * wq) << 16) + a * D + 32 * j, v);
                    tmem_wait_ld();
                    unsigned char* hb = st + (j / 2) * (kLtRows * 128) + m * 128;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int chunk = ((32 * j) % 64) / 8 + q;
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
            if (lane == 0) mbar_arrive(&tempty[a]);
            fence_proxy_async_smem();  // epilogue writes -> TMA store reads
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et == 0) {
                if (ok) {
                    const int t0 = (tile0 + i) * kLtRows;
                    for (int half = 0; half < D / 64; ++half)
                        tma_store_4d(&tm_out, st + half * (kLtRows * 128), h * D + 64 * half, t0, l, c);
                }
                bulk_commit();
                bulk_wait_read<1>();  // the previous tile's store has read its stage
                if (i >= 1) mbar_arrive(&empty[(i - 1) % kLtStages]);
            }
            if (!ok) break;
        }
        if (et == 0) bulk_wait<0>();
    }
    __syncthreads();
    if (abort_flag && threadIdx.x == 0) atomicOr(&g_status_lowrank, FLAG_TIMEOUT);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::kCols);
}

static cudaError_t encode_plane(CUtensorMap* map, const void* base, const Plane& p) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[4], strides[3];
    plane_map_strides(p, dims, strides);
    cuuint32_t box[4] = {64, (cuuint32_t)kLtRows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int RANK>
static cudaError_t launch_lowrank_t(const uint16_t* x, const Plane& p, const uint16_t* A, const uint16_t* B,
                                    uint16_t* out, const Plane& op, cudaStream_t s) {
    using C = LtCfg<D, RANK>;
    CUtensorMap tx, to, ta;
    cudaError_t e;
    if ((e = encode_plane(&tx, x, p)) != cudaSuccess) return e;
    if ((e = encode_plane(&to, out, op)) != cudaSuccess) return e;
    auto enc = tensor_map_encoder();
    const long long rows = (long long)p.chunks * p.layers * p.heads * p.tokens;
    cuuint64_t adims[2] = {(cuuint64_t)RANK, (cuuint64_t)rows};
    cuuint64_t astr[1] = {(cuuint64_t)RANK * 2};
    cuuint32_t abox[2] = {(cuuint32_t)RANK, (cuuint32_t)kLtRows};
    cuuint32_t aestr[2] = {1, 1};
    if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A), adims, astr, abox, aestr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(C::kASwizzleBytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    LtArgs args;
    args.B = B;
    args.H = p.heads;
    args.L = p.layers;
    args.n = p.tokens;
    args.tiles_per_unit = (p.tokens + kLtRows - 1) / kLtRows;
    args.tiles_per_cta = kLtTilesPerCta;
    e = cudaFuncSetAttribute(lowrank_tc_kernel<D, RANK>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((args.tiles_per_unit + kLtTilesPerCta - 1) / kLtTilesPerCta, p.heads, p.chunks * p.layers);
    lowrank_tc_kernel<D, RANK><<<grid, kLtThreads, C::kSmem, s>>>(tx, to, ta, args);
    return cudaGetLastError();
}

cudaError_t launch_lowrank(const uint16_t* x, const kvfix_kv_desc& d, const uint16_t* A,
                           const uint16_t* B, int rank, uint16_t* out, const kvfix_kv_desc& od,
                           cudaStream_t s) {
    Plane p = plane_of(d), op = plane_of(od);
    if (p.chunks == 0 || p.layers == 0 || p.tokens == 0) return cudaSuccess;
    if (p.dim == 128) {
        if (rank == 16) return launch_lowrank_t<128, 16>(x, p, A, B, out, op, s);
        if (rank == 32) return launch_lowrank_t<128, 32>(x, p, A, B, out, op, s);
        return launch_lowrank_t<128, 64>(x, p, A, B, out, op, s);
    }
    if (rank == 16) return launch_lowrank_t<64, 16>(x, p, A, B, out, op, s);
    if (rank == 32) return launch_lowrank_t<64, 32>(x, p, A, B, out, op, s);
    return launch_lowrank_t<64, 64>(x, p, A, B, out, op, s);
}

}  // namespace kvfix
