// Projection GEMM on tcgen05 tensor cores (sm_103a): C[M, N] = A[M, K] W[N, K]^T,
// bf16 in, fp32 accumulation in tensor memory, bf16 or fp32 out.
//
// The projections on either side of attention (TSP summary, "Folding Tensor
// and Sequence Parallelism", section 2, attention layer: every rank computes
// the local projections of its sequence shard with each packed W_Q, W_K, W_V,
// W_O shard in turn).  On one GPU the sequence shards are row ranges of one
// buffer and the weight shards column ranges of one weight, so the union of
// all (sequence shard x weight shard) products is this one GEMM over all rows
// in buffer order.
//
// Persistent kernel: one CTA per SM walks the 128 x 256 output tiles in
// groups of row blocks (tile_coords), so the CTAs working at one time share
// a few row blocks of A and a few column blocks of W in L2 even when W is
// larger than L2.  Warp roles (192 threads):
//   warp 0     TMA producer: 64-wide K blocks of A (128 rows) and W (256 rows)
//              into a 4-stage shared-memory ring;
//   warp 1     TMEM allocator and single-thread MMA issuer: 4 MMAs
//              (M = 128, N = 256, K = 16) per K block into one of two TMEM
//              accumulators (2 x 256 columns), so the epilogue of one tile
//              overlaps the MMAs of the next;
//   warps 2-5  epilogue: one accumulator row per thread, TMEM -> registers ->
//              bf16 / fp32 -> global memory (rows and columns past M, N are
//              not stored; K past the end is zero-filled by the TMA).
// Every barrier wait is bounded (tc_ptx.cuh).
//
// Gated variant (the gate and up projections of a gated MLP, TSP summary,
// section 2, gated MLP layer): the 256 rows of the W tile are 128 rows of W1
// followed by the same 128 rows of W3, so one MMA tile holds the gate
// a = x W1^T and the up value b = x W3^T for 128 hidden units side by side,
// and the epilogue writes h = silu(a) * b (bf16) for those 128 columns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "tc_ptx.cuh"

namespace st {
namespace {

using namespace tc;

constexpr int kGM = 128;          // rows per tile (MMA M)
constexpr int kGN = 256;          // columns per tile (MMA N)
constexpr int kGK = 64;           // K per block: one 128-byte swizzle atom of bf16
constexpr int kGStages = 4;
constexpr int kGThreads = 192;
constexpr int kABytes = kGM * kGK * 2;   // 16 KB
constexpr int kWBytes = kGN * kGK * 2;   // 32 KB
constexpr int kGAOff = 0;
constexpr int kGWOff = kGAOff + kGStages * kABytes;
constexpr int kGBarOff = kGWOff + kGStages * kWBytes;
// full[S], empty[S], acc_full[2], acc_empty[2], drain
constexpr int kGNumBars = 2 * kGStages + 5;
constexpr int kGMiscOff = kGBarOff + kGNumBars * 8;
constexpr int kGSmemBytes = kGMiscOff + 16 + 1024;
static_assert(kGSmemBytes <= 232448, "shared memory per CTA");

// Output tile t -> (row block, column block).  Tiles are taken in groups of
// `group` row blocks; inside a group the column block is the slow index.  The
// CTAs working at one time then share a few row blocks of A and a few column
// blocks of W, both small enough to stay in L2, instead of all of W.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group, int& mb, int& nb) {
    const int per_group = group * tiles_n;
    const int g = t / per_group, local = t % per_group;
    const int gm = min(group, tiles_m - g * group);
    mb = g * group + local % gm;
    nb = local / gm;
}

struct GemmParams {
    CUtensorMap ta;     // A: (K, M) bf16, box (64, 128), 128-byte swizzle
    CUtensorMap tw;     // W: (K, N) bf16, box (64, 256); gated: W1, box (64, 128)
    CUtensorMap tw3;    // gated only: W3 (K, N) bf16, box (64, 128)
    void* c;            // [M, N] bf16 or fp32 (gated: h, bf16)
    int M, N, K;
    int out_f32;
    int group;          // row blocks per tile group (tile_coords)
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// x * sigmoid(x), with the exponential from the CUDA intrinsic; exp(-x) = inf
// for very negative x gives -0, the limit.
__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

template <bool kGated>
__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    constexpr int kTN = kGated ? kGN / 2 : kGN;   // output columns per tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t sA = sbase + kGAOff, sW = sbase + kGWOff;
    const uint32_t bars = sbase + kGBarOff;
    auto bar_full = [&](int s) { return bars + 8u * s; };
    auto bar_empty = [&](int s) { return bars + 8u * (kGStages + s); };
    auto bar_accf = [&](int a) { return bars + 8u * (2 * kGStages + a); };
    auto bar_acce = [&](int a) { return bars + 8u * (2 * kGStages + 2 + a); };
    const uint32_t bar_drain = bars + 8u * (2 * kGStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kGMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kGMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_m = (p.M + kGM - 1) / kGM, tiles_n = (p.N + kTN - 1) / kTN;
    const int ntiles = tiles_m * tiles_n;
    const int nkb = (p.K + kGK - 1) / kGK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_accf(a), 1);
            mbar_init(bar_acce(a), 128);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.ta);
        prefetch_tmap(&p.tw);
        if (kGated) prefetch_tmap(&p.tw3);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;   // K blocks issued so far (over all tiles)
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, tiles_m, tiles_n, p.group, mb, nb);
                const int m0 = mb * kGM, n0 = nb * kTN;
                for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                    const int s = it % kGStages;
                    if (it >= kGStages) ok = mbar_wait(bar_empty(s), ((it / kGStages) - 1) & 1, abort_flag);
                    if (!ok) break;
                    // both gated boxes are full 128-row boxes (rows past N zero-filled)
                    mbar_arrive_expect_tx(bar_full(s), kABytes + kWBytes);
                    tma_load_2d(sA + s * kABytes, &p.ta, bar_full(s), kb * kGK, m0);
                    tma_load_2d(sW + s * kWBytes, &p.tw, bar_full(s), kb * kGK, n0);
                    if (kGated) tma_load_2d(sW + s * kWBytes + kWBytes / 2, &p.tw3, bar_full(s), kb * kGK, n0);
                }
            }
            // every load issued lands before the CTA can exit (also after an abort)
            for (int i = max(0, it - kGStages); i < it; ++i)
                mbar_wait_drain(bar_full(i % kGStages), (i / kGStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN, 0, 0);
            const uint64_t adesc = smem_desc_sw128(sA, 16, 1024);
            const uint64_t wdesc = smem_desc_sw128(sW, 16, 1024);
            int it = 0, nt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++nt) {
                const int a = nt & 1;
                // the epilogue has emptied this accumulator (used two tiles ago)
                if (nt >= 2) ok = mbar_wait(bar_acce(a), ((nt >> 1) - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(a * kGN);
                for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                    const int s = it % kGStages;
                    ok = mbar_wait(bar_full(s), (it / kGStages) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t ad = adesc + (uint64_t)(s * (kABytes >> 4));
                    const uint64_t wd = wdesc + (uint64_t)(s * (kWBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk)
                        mma_ss(acc, ad + (uint64_t)(kk * 2), wd + (uint64_t)(kk * 2), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar_empty(s));
                }
                if (ok) mma_commit(bar_accf(a));
            }
            mma_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                       // accumulator row
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        int nt = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++nt) {
            const int a = nt & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_accf(a), (nt >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            int mb, nb;
            tile_coords(tile, tiles_m, tiles_n, p.group, mb, nb);
            const int row = mb * kGM + r, n0 = nb * kTN;
            if constexpr (kGated) {
#pragma unroll 1
                for (int c = 0; c < kTN / 32; ++c) {
                    uint32_t ga[32], up[32];
                    tmem_ld32(lane_base + (uint32_t)(a * kGN + c * 32), ga);
                    tmem_ld32(lane_base + (uint32_t)(a * kGN + kTN + c * 32), up);
                    tmem_wait_ld();
                    const int col = n0 + c * 32;
                    if (row < p.M && col < p.N) {
                        const int ngrp = min(4, (p.N - col) / 8);
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.c) + (int64_t)row * p.N + col;
                        float h[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) h[i] = silu(__uint_as_float(ga[i])) * __uint_as_float(up[i]);
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            if (g < ngrp)
                                *reinterpret_cast<uint4*>(dst + 8 * g) =
                                    make_uint4(pack_bf16x2(h[8 * g], h[8 * g + 1]), pack_bf16x2(h[8 * g + 2], h[8 * g + 3]),
                                               pack_bf16x2(h[8 * g + 4], h[8 * g + 5]),
                                               pack_bf16x2(h[8 * g + 6], h[8 * g + 7]));
                    }
                }
                tc_fence_before();
                mbar_arrive(bar_acce(a));
                continue;
            }
#pragma unroll 1
            for (int c = 0; c < kGN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_base + (uint32_t)(a * kGN + c * 32), v);
                tmem_wait_ld();
                const int col = n0 + c * 32;
                if (row < p.M && col < p.N) {
                    // N is a multiple of 8: whole groups of 8 columns are stored
                    const int ngrp = min(4, (p.N - col) / 8);
                    if (p.out_f32) {
                        float* dst = static_cast<float*>(p.c) + (int64_t)row * p.N + col;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            if (g < ngrp) {
                                reinterpret_cast<float4*>(dst + 8 * g)[0] =
                                    make_float4(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1]),
                                                __uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                                reinterpret_cast<float4*>(dst + 8 * g)[1] =
                                    make_float4(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]),
                                                __uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
                            }
                    } else {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.c) + (int64_t)row * p.N + col;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            if (g < ngrp)
                                *reinterpret_cast<uint4*>(dst + 8 * g) = make_uint4(
                                    pack_bf16x2(__uint_as_float(v[8 * g]), __uint_as_float(v[8 * g + 1])),
                                    pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3])),
                                    pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5])),
                                    pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])));
                    }
                }
            }
            // the accumulator may be overwritten by the tile after next
            tc_fence_before();
            mbar_arrive(bar_acce(a));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Row-major bf16 [rows, K] as a 2-D map (K, rows), box (64, box_rows), 128-byte
// swizzle; out-of-range elements are read as zero.
bool make_map_2d(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGated>
int launch(GemmParams p, void* stream) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    const int tn = kGated ? kGN / 2 : kGN;
    const int tiles_m = (p.M + kGM - 1) / kGM;
    const int ntiles = tiles_m * ((p.N + tn - 1) / tn);
    // A W of at most 32 MB stays in L2 whole: take the tiles row block by row
    // block (group 1), so that the CTAs working at one time share A rows.  A
    // larger W is taken in groups of row blocks whose A rows (kGM x K bf16
    // each) fit in 32 MB, column block by column block within the group.
    const int64_t w_bytes = (int64_t)p.N * p.K * 2;
    const int64_t a_block = (int64_t)kGM * p.K * 2;
    int64_t group = w_bytes <= ((int64_t)32 << 20) ? 1 : ((int64_t)32 << 20) / a_block;
    p.group = (int)(group < 1 ? 1 : (group > tiles_m ? tiles_m : group));
    const int grid = ntiles < sms ? ntiles : sms;
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel<kGated>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmemBytes);
    if (e != cudaSuccess) return (int)e;
    gemm_tc_kernel<kGated><<<grid, kGThreads, kGSmemBytes, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_gemm_tc(int M, int N, int K, const void* a, const void* w, void* c, int out_dtype, void* stream) {
    GemmParams p;
    if (!make_map_2d(&p.ta, a, M, K, kGM) || !make_map_2d(&p.tw, w, N, K, kGN)) return (int)cudaErrorInvalidValue;
    p.tw3 = p.tw;
    p.c = c;
    p.M = M;
    p.N = N;
    p.K = K;
    p.out_f32 = out_dtype == ST_DTYPE_F32 ? 1 : 0;
    return launch<false>(p, stream);
}

int launch_gemm_gated(int M, int F, int K, const void* a, const void* w1, const void* w3, void* h, void* stream) {
    GemmParams p;
    if (!make_map_2d(&p.ta, a, M, K, kGM) || !make_map_2d(&p.tw, w1, F, K, kGN / 2) ||
        !make_map_2d(&p.tw3, w3, F, K, kGN / 2))
        return (int)cudaErrorInvalidValue;
    p.c = h;
    p.M = M;
    p.N = F;
    p.K = K;
    p.out_f32 = 0;
    return launch<true>(p, stream);
}

int gemm_tc_device_error(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(tc::g_device_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace st
