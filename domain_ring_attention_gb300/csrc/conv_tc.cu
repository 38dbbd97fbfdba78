// Halo exchange and 2-D convolution of a row-sharded image (sm_103a).
//
// ShardTensor summary, "ShardTensor" section 2, implementation details,
// communication.  A convolution over an input whose spatial axes are split
// over devices needs the neighbouring pixels that the adjacent chunks hold
// (the "halo") to give the numbers of the layer on the whole input.  The
// chunks may be uneven (section 2, sharding shapes).
//
// Layout: shard r is its own buffer, as it would be on its own device,
// channels last and padded by h = (k - 1) / 2 rows on each side:
//   x_r [L_r + 2h, W, C_in] bf16.
// Rows h .. h + L_r - 1 hold the shard's image rows off_r .. off_r + L_r - 1.
//
//   halo_kernel     fills the 2h pad rows of every shard from the shards that
//                   own those image rows (zero outside the image).  With
//                   several GPUs these would be peer copies; here they are
//                   device-local copies.
//   conv_tc_kernel  y_r[i, j, o] = bias[o] + sum_{u,v,c} x_r[i + u, j + v - h, c] w[o, u, v, c]
//                   (a cross-correlation, zero outside the image along W) as an implicit GEMM on tcgen05:
//                   M = 128 pixels of one output row, N = up to 256 output channels,
//                   K = k*k*C_in walked tap by tap in blocks of 64 channels.
//                   For tap (u, v) and channel block cb, the A tile is a 3-D TMA box
//                   (64 channels x 128 pixels x 1 row) at (cb*64, x0 + v - h, i + u) of
//                   the shard's padded buffer.  Pixels left of 0 or right of W - 1 are
//                   zero-filled by the TMA, which gives the W padding without an
//                   im2col buffer.  The B tile is the weight slice [n0 .. n0 + N) x
//                   (tap, cb): the weight is [C_out, k, k, C_in], i.e. row-major
//                   [C_out, K].
//
// Persistent CTAs: one per SM, walking (image row, pixel tile, channel tile)
// units with the channel tile fastest.  The CTAs working at one time read
// neighbouring rows, which stay in L2.  Warp roles as in the projection GEMM:
//   warp 0: TMA producer (4-stage ring);
//   warp 1: TMEM and the single MMA issuer, with two accumulators;
//   warps 2-5: epilogue (bias, bf16 / fp32 stores).
// Every barrier wait is bounded (tc_ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "common.h"
#include "tc_ptx.cuh"

namespace st {
namespace {

using namespace tc;

constexpr int kMaxShards = ST_CONV_MAX_SHARDS;   // one tensor map per shard in the kernel parameters
constexpr int kCM = 128;          // pixels per tile (MMA M)
constexpr int kCNMax = 256;       // output channels per tile at most (MMA N)
constexpr int kCK = 64;           // channels per K block (one 128-byte swizzle atom)
constexpr int kCStages = 4;
constexpr int kCThreads = 192;
constexpr int kCABytes = kCM * kCK * 2;      // 16 KB
constexpr int kCWBytes = kCNMax * kCK * 2;   // 32 KB (the largest channel tile)
constexpr int kCAOff = 0;
constexpr int kCWOff = kCAOff + kCStages * kCABytes;
constexpr int kCBarOff = kCWOff + kCStages * kCWBytes;
constexpr int kCNumBars = 2 * kCStages + 5;  // full[S], empty[S], acc_full[2], acc_empty[2], drain
constexpr int kCMiscOff = kCBarOff + kCNumBars * 8;
constexpr int kCSmemBytes = kCMiscOff + 16 + 1024;
static_assert(kCSmemBytes <= 232448, "shared memory per CTA");

struct ConvParams {
    CUtensorMap tin[kMaxShards];   // shard r: (C_in, W, L_r + 2h) bf16, box (64, 128, 1), 128-byte swizzle
    CUtensorMap tw;                // weight: (k*k*C_in, C_out) bf16, box (64, n_tile)
    void* out[kMaxShards];         // shard r: [L_r, W, C_out]
    const float* bias;             // [C_out] or null
    int off[kMaxShards + 1];       // image row of each shard's first row
    int D, W, C_in, C_out, k;
    int n_tile, tiles_x, tiles_n;
    int out_f32;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_c(uint32_t dst, const void* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// image row g -> (shard, row within the shard); D <= kMaxShards
__device__ __forceinline__ int owner(const int* off, int D, int g) {
    int r = 0;
    while (r + 1 < D && off[r + 1] <= g) ++r;
    return r;
}

__global__ void __launch_bounds__(kCThreads, 1) conv_tc_kernel(const __grid_constant__ ConvParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t sA = sbase + kCAOff, sW = sbase + kCWOff;
    const uint32_t bars = sbase + kCBarOff;
    auto bar_full = [&](int s) { return bars + 8u * s; };
    auto bar_empty = [&](int s) { return bars + 8u * (kCStages + s); };
    auto bar_accf = [&](int a) { return bars + 8u * (2 * kCStages + a); };
    auto bar_acce = [&](int a) { return bars + 8u * (2 * kCStages + 2 + a); };
    const uint32_t bar_drain = bars + 8u * (2 * kCStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kCMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kCMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.off[p.D];
    const int per_row = p.tiles_x * p.tiles_n;
    const int nunits = H * per_row;
    const int cblocks = p.C_in / kCK;
    const int nkb = p.k * p.k * cblocks;
    const int h = (p.k - 1) / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCStages; ++s) {
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
    if (warp == 0 && lane < p.D) prefetch_tmap(&p.tin[lane]);
    if (warp == 0 && lane == 0) prefetch_tmap(&p.tw);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t tx = kCABytes + (uint32_t)p.n_tile * kCK * 2;
            int it = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < nunits && ok; unit += gridDim.x) {
                const int g = unit / per_row, rem = unit % per_row;
                const int x0 = (rem / p.tiles_n) * kCM, n0 = (rem % p.tiles_n) * p.n_tile;
                const int r = owner(p.off, p.D, g);
                const int i = g - p.off[r];          // output row within the shard = padded row of tap u = 0
                const void* tin = &p.tin[r];
                for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                    const int tap = kb / cblocks, cb = kb % cblocks;
                    const int u = tap / p.k, v = tap % p.k;
                    const int s = it % kCStages;
                    if (it >= kCStages) ok = mbar_wait(bar_empty(s), ((it / kCStages) - 1) & 1, abort_flag);
                    if (!ok) break;
                    // full boxes: pixels outside 0 .. W-1 and channels past C_out arrive as zeros
                    mbar_arrive_expect_tx(bar_full(s), tx);
                    tma_load_3d(sA + s * kCABytes, tin, bar_full(s), cb * kCK, x0 + v - h, i + u);
                    tma_load_2d_c(sW + s * kCWBytes, &p.tw, bar_full(s), tap * p.C_in + cb * kCK, n0);
                }
            }
            for (int q = max(0, it - kCStages); q < it; ++q)
                mbar_wait_drain(bar_full(q % kCStages), (q / kCStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kCM, p.n_tile, 0, 0);
            const uint64_t adesc = smem_desc_sw128(sA, 16, 1024);
            const uint64_t wdesc = smem_desc_sw128(sW, 16, 1024);
            int it = 0, nt = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < nunits && ok; unit += gridDim.x, ++nt) {
                const int a = nt & 1;
                if (nt >= 2) ok = mbar_wait(bar_acce(a), ((nt >> 1) - 1) & 1, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(a * kCNMax);
                for (int kb = 0; kb < nkb && ok; ++kb, ++it) {
                    const int s = it % kCStages;
                    ok = mbar_wait(bar_full(s), (it / kCStages) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t ad = adesc + (uint64_t)(s * (kCABytes >> 4));
                    const uint64_t wd = wdesc + (uint64_t)(s * (kCWBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kCK / 16; ++kk)
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
        const int pix = quad * 32 + lane;                     // accumulator row = pixel in the tile
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        int nt = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < nunits && ok; unit += gridDim.x, ++nt) {
            const int a = nt & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_accf(a), (nt >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int g = unit / per_row, rem = unit % per_row;
            const int x = (rem / p.tiles_n) * kCM + pix, n0 = (rem % p.tiles_n) * p.n_tile;
            const int r = owner(p.off, p.D, g);
            const int64_t prow = (int64_t)(g - p.off[r]) * p.W + x;      // pixel index within shard r's output
#pragma unroll 1
            for (int c = 0; c < p.n_tile; c += 32) {
                uint32_t v[32];
                tmem_ld32(lane_base + (uint32_t)(a * kCNMax + c), v);
                tmem_wait_ld();
                const int col = n0 + c;
                if (x < p.W && col < p.C_out) {
                    const int ngrp = min(min(4, (p.C_out - col) / 8), (p.n_tile - c) / 8);
                    float f[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) f[q] = __uint_as_float(v[q]);
                    if (p.bias) {
#pragma unroll
                        for (int q = 0; q < 32; ++q)
                            if (q < 8 * ngrp) f[q] += __ldg(p.bias + col + q);
                    }
                    if (p.out_f32) {
                        float* dst = static_cast<float*>(p.out[r]) + prow * p.C_out + col;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < ngrp) {
                                reinterpret_cast<float4*>(dst + 8 * q)[0] =
                                    make_float4(f[8 * q], f[8 * q + 1], f[8 * q + 2], f[8 * q + 3]);
                                reinterpret_cast<float4*>(dst + 8 * q)[1] =
                                    make_float4(f[8 * q + 4], f[8 * q + 5], f[8 * q + 6], f[8 * q + 7]);
                            }
                    } else {
                        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[r]) + prow * p.C_out + col;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < ngrp)
                                *reinterpret_cast<uint4*>(dst + 8 * q) =
                                    make_uint4(pack2_bf16(f[8 * q], f[8 * q + 1]), pack2_bf16(f[8 * q + 2], f[8 * q + 3]),
                                               pack2_bf16(f[8 * q + 4], f[8 * q + 5]),
                                               pack2_bf16(f[8 * q + 6], f[8 * q + 7]));
                    }
                }
            }
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

// ---------------------------------------------------------------- halo exchange

struct HaloParams {
    void* shard[kMaxShards];       // shard r: [L_r + 2h, W, C] bf16
    int off[kMaxShards + 1];
    int D, h;
    int64_t row_vec;               // 16-byte vectors per image row: W * C / 8
};

// One thread per 16-byte vector of a pad row; the 2h pad rows of every shard
// in turn.  Reads touch only shards' own rows, writes only pad rows.
__global__ void halo_kernel(const __grid_constant__ HaloParams p) {
    const int64_t per_shard = 2 * (int64_t)p.h * p.row_vec;
    const int64_t total = per_shard * p.D;
    const int H = p.off[p.D];
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(idx / per_shard);
        const int64_t rem = idx % per_shard;
        const int pr = (int)(rem / p.row_vec);                  // pad row 0 .. 2h-1
        const int64_t e = rem % p.row_vec;
        const int L = p.off[r + 1] - p.off[r];
        const int dst_row = pr < p.h ? pr : L + pr;               // padded row index
        const int g = p.off[r] - p.h + dst_row;                   // its image row
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (g >= 0 && g < H) {
            const int s = owner(p.off, p.D, g);
            const uint4* src = static_cast<const uint4*>(p.shard[s]);
            val = src[(int64_t)(p.h + g - p.off[s]) * p.row_vec + e];
        }
        static_cast<uint4*>(p.shard[r])[(int64_t)dst_row * p.row_vec + e] = val;
    }
}

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

int num_sms() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return sms;
}

}  // namespace

int launch_halo_exchange(int D, const int64_t* rows, int W, int C, int h, void* const* shards, void* stream) {
    if (h == 0) return 0;
    HaloParams p;
    p.off[0] = 0;
    for (int r = 0; r < D; ++r) {
        p.shard[r] = shards[r];
        p.off[r + 1] = p.off[r] + (int)rows[r];
    }
    p.D = D;
    p.h = h;
    p.row_vec = (int64_t)W * C / 8;
    const int64_t total = 2 * (int64_t)h * p.row_vec * D;
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)num_sms() * 8 ? want : (int64_t)num_sms() * 8);
    halo_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

int launch_conv_tc(int D, const int64_t* rows, int W, int C_in, int C_out, int k, void* const* in_shards,
                   const void* weight, const float* bias, void* const* out_shards, int out_dtype, void* stream) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return (int)cudaErrorInvalidValue;
    ConvParams p;
    const int h = (k - 1) / 2;
    p.n_tile = C_out >= kCNMax ? kCNMax : ((C_out + 15) / 16) * 16;
    p.off[0] = 0;
    for (int r = 0; r < D; ++r) {
        const cuuint64_t dims[3] = {(cuuint64_t)C_in, (cuuint64_t)W, (cuuint64_t)(rows[r] + 2 * h)};
        const cuuint64_t strides[2] = {(cuuint64_t)C_in * 2, (cuuint64_t)W * C_in * 2};
        const cuuint32_t box[3] = {(cuuint32_t)kCK, (cuuint32_t)kCM, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc(&p.tin[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, in_shards[r], dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return (int)cudaErrorInvalidValue;
        p.out[r] = out_shards[r];
        p.off[r + 1] = p.off[r] + (int)rows[r];
    }
    for (int r = D; r < kMaxShards; ++r) {
        p.tin[r] = p.tin[0];
        p.out[r] = nullptr;
        p.off[r + 1] = p.off[D];
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)k * k * C_in, (cuuint64_t)C_out};
        const cuuint64_t strides[1] = {(cuuint64_t)k * k * C_in * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kCK, (cuuint32_t)p.n_tile};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&p.tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(weight), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return (int)cudaErrorInvalidValue;
    }
    p.bias = bias;
    p.D = D;
    p.W = W;
    p.C_in = C_in;
    p.C_out = C_out;
    p.k = k;
    p.tiles_x = (W + kCM - 1) / kCM;
    p.tiles_n = (C_out + p.n_tile - 1) / p.n_tile;
    p.out_f32 = out_dtype == ST_DTYPE_F32 ? 1 : 0;
    const int64_t nunits = (int64_t)p.off[D] * p.tiles_x * p.tiles_n;
    const int grid = (int)(nunits < num_sms() ? nunits : num_sms());
    cudaError_t e = cudaFuncSetAttribute(conv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmemBytes);
    if (e != cudaSuccess) return (int)e;
    conv_tc_kernel<<<grid, kCThreads, kCSmemBytes, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

int conv_tc_device_error(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(tc::g_device_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace st
