// Bandwidth-bound helper kernels: the standalone log-sum-exp merge, the
// backward row sums Delta, the dQ accumulator conversion and the
// buffer <-> natural row permutation.
//
// All four stream rows of d contiguous elements (the merge with 4 elements
// per thread, the others one warp per row with lanes moving consecutive
// 8/16-byte pieces), in grid-stride loops over rows with the grid sized to a
// multiple of the SM count.
#include <cmath>

#include <cuda_fp16.h>

#include "device.cuh"

namespace st {
namespace {

constexpr int kWarps = 8;

int grid_for(int64_t rows) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    const int64_t want = (rows + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)sms * 16;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

// Log-sum-exp merge (ring-attention combine): L = log sum_j exp(lse_j),
// out = sum_j exp(lse_j - L) O_j; every lse_j = -inf gives L = -inf, out = 0.
// Each thread owns 4 consecutive elements of a row (16 threads per row at
// d = 64, 32 at d = 128) and issues the loads of kBatch partials before it
// combines them, so that enough bytes are in flight to keep HBM busy (one
// dependent load per partial and warp left the kernel latency-bound).
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
merge_kernel(int nparts, int B, int H, int S, const float* __restrict__ part_out,
             const float* __restrict__ part_lse, T* __restrict__ out, float* __restrict__ lse) {
    constexpr int TPR = D / 4;     // threads per row
    constexpr int RPW = 32 / TPR;  // rows per warp
    constexpr int kBatch = 8;      // partials whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const int c4 = lane % TPR;
    const int64_t nrows = (int64_t)B * S * H;
    const int64_t elems = nrows * D;
    const int64_t lse_n = (int64_t)B * H * S;
    const int64_t stride = (int64_t)gridDim.x * kWarps * RPW;
    for (int64_t row = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * RPW + lane / TPR; row < nrows;
         row += stride) {
        const int h = (int)(row % H);
        const int64_t bs = row / H;
        const int s = (int)(bs % S);
        const int b = (int)(bs / S);
        const int64_t li = ((int64_t)b * H + h) * S + s;
        float m = -INFINITY;
        for (int j = 0; j < nparts; ++j) m = fmaxf(m, __ldg(part_lse + j * lse_n + li));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float tot = 0.f;
        if (m != -INFINITY) {
            for (int j0 = 0; j0 < nparts; j0 += kBatch) {
                float4 x[kBatch];
                float l[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int j = j0 + u;
                    if (j < nparts) {
                        x[u] = __ldcs(reinterpret_cast<const float4*>(part_out + j * elems + row * D) + c4);
                        l[u] = __ldg(part_lse + j * lse_n + li);
                    } else {
                        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        l[u] = -INFINITY;
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (j0 + u < nparts) {
                        const float w = expf(l[u] - m);
                        tot += w;
                        acc.x = fmaf(w, x[u].x, acc.x);
                        acc.y = fmaf(w, x[u].y, acc.y);
                        acc.z = fmaf(w, x[u].z, acc.z);
                        acc.w = fmaf(w, x[u].w, acc.w);
                    }
                }
            }
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
        T* dst = out + row * D + c4 * 4;
        if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        }
        if (c4 == 0) lse[li] = tot > 0.f ? m + logf(tot) : -INFINITY;
    }
}

// N consecutive elements (N = 2 or 4, 4N- or 2N-byte aligned) as floats, one vector load.
template <int N>
__device__ __forceinline__ void load_vec(const float* p, float (&x)[N]) {
    if constexpr (N == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x; x[1] = v.y;
    }
}
template <int N>
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&x)[N]) {
    if constexpr (N == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        x[0] = a.x; x[1] = a.y; x[2] = c.x; x[3] = c.y;
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
        x[0] = a.x; x[1] = a.y;
    }
}

// Delta_i = sum_c dO_ic * O_ic in fp32 (backward preprocess).  A warp takes 32
// consecutive positions s of one (b, h): each row is read as one contiguous
// vector per lane (four rows in flight before any is reduced), lane r keeps
// the sum of row r, and the 32 sums go out as one coalesced store into
// Delta[b, h, s0 .. s0+31] (Delta is [B, H, S], the rows [B, S, H]).
template <typename TO, typename T, int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
delta_kernel(int B, int H, int S, const TO* __restrict__ o, const T* __restrict__ dout,
             float* __restrict__ delta) {
    constexpr int PER = D / 32;
    constexpr int R = 4;   // rows in flight per warp
    const int lane = threadIdx.x & 31;
    const int sblocks = (S + 31) / 32;
    const int64_t nunits = (int64_t)B * H * sblocks;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); u < nunits;
         u += (int64_t)gridDim.x * kWarps) {
        const int sb = (int)(u % sblocks);
        const int64_t bh = u / sblocks;
        const int h = (int)(bh % H);
        const int b = (int)(bh / H);
        const int s0 = sb * 32;
        float mine = 0.f;
#pragma unroll 1
        for (int r0 = 0; r0 < 32; r0 += R) {
            float vo[R][PER], vg[R][PER];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int s = s0 + r0 + r;
                if (s < S) {
                    const int64_t row = ((int64_t)b * S + s) * H + h;
                    load_vec<PER>(o + row * D + lane * PER, vo[r]);
                    load_vec<PER>(dout + row * D + lane * PER, vg[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float acc = 0.f;
                if (s0 + r0 + r < S) {
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc = fmaf(vo[r][e], vg[r][e], acc);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (lane == r0 + r) mine = acc;
            }
        }
        if (s0 + lane < S) delta[bh * S + s0 + lane] = mine;
    }
}

template <typename T>
__global__ void convert_kernel(int64_t n, const float* __restrict__ src, T* __restrict__ dst) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = from_f32<T>(src[i]);
}

// Row permutation between buffer order and natural order, 16-byte pieces.
__global__ void __launch_bounds__(kWarps * 32)
permute_kernel(const __grid_constant__ SegTable tab, int B, int H, int row_bytes,
               int to_natural, const uint4* __restrict__ in, uint4* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int pieces = row_bytes / 16;
    const int S = tab.S;
    const int64_t nrows = (int64_t)B * S;
    for (int64_t bt = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); bt < nrows;
         bt += (int64_t)gridDim.x * kWarps) {
        const int t = (int)(bt % S);
        const int64_t b = bt / S;
        int s = 0;
        while (s + 1 < tab.nseg && tab.seg_buf[s + 1] <= t) ++s;
        const int p = tab.seg_nat[s] + (t - tab.seg_buf[s]);
        const int64_t src_row = b * S + (to_natural ? t : p);
        const int64_t dst_row = b * S + (to_natural ? p : t);
        const int64_t per_tok = (int64_t)H * pieces;
        for (int64_t i = lane; i < per_tok; i += 32) out[dst_row * per_tok + i] = in[src_row * per_tok + i];
    }
}

}  // namespace

int launch_merge(int D, int B, int H, int64_t S, int d, const float* part_out,
                 const float* part_lse, void* out, float* lse, int out_dtype, void* stream) {
    const int64_t rows = (int64_t)B * S * H;
    const int grid = grid_for(rows);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (out_dtype == ST_DTYPE_F32) {
        if (d == 64)
            merge_kernel<float, 64><<<grid, kWarps * 32, 0, st>>>(D, B, H, (int)S, part_out, part_lse,
                                                                  static_cast<float*>(out), lse);
        else
            merge_kernel<float, 128><<<grid, kWarps * 32, 0, st>>>(D, B, H, (int)S, part_out, part_lse,
                                                                   static_cast<float*>(out), lse);
    } else {
        if (d == 64)
            merge_kernel<__nv_bfloat16, 64><<<grid, kWarps * 32, 0, st>>>(
                D, B, H, (int)S, part_out, part_lse, static_cast<__nv_bfloat16*>(out), lse);
        else
            merge_kernel<__nv_bfloat16, 128><<<grid, kWarps * 32, 0, st>>>(
                D, B, H, (int)S, part_out, part_lse, static_cast<__nv_bfloat16*>(out), lse);
    }
    return (int)cudaGetLastError();
}

int launch_bwd_preprocess(const BwdArgs& a, int64_t S, int dtype, void* stream) {
    const int64_t rows = (int64_t)a.B * S * a.H;
    const int grid = grid_for(rows);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    using bf16 = __nv_bfloat16;
    if (dtype == ST_DTYPE_F32) {
        auto o = static_cast<const float*>(a.out);
        auto g = static_cast<const float*>(a.dout);
        if (a.d == 64)
            delta_kernel<float, float, 64><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
        else
            delta_kernel<float, float, 128><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
    } else if (a.out_dtype == ST_DTYPE_F32) {
        auto o = static_cast<const float*>(a.out);
        auto g = static_cast<const bf16*>(a.dout);
        if (a.d == 64)
            delta_kernel<float, bf16, 64><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
        else
            delta_kernel<float, bf16, 128><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
    } else {
        auto o = static_cast<const bf16*>(a.out);
        auto g = static_cast<const bf16*>(a.dout);
        if (a.d == 64)
            delta_kernel<bf16, bf16, 64><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
        else
            delta_kernel<bf16, bf16, 128><<<grid, kWarps * 32, 0, st>>>(a.B, a.H, (int)S, o, g, a.delta);
    }
    return (int)cudaGetLastError();
}

namespace {

// ---- exact fp16 operand copies for the tensor-core backward ----
//
// bf16 carries 8 significant bits and fp16 11, so a bf16 value times a power
// of two is exactly representable in fp16 as long as it lands in fp16's normal
// range.  Each tensor is scaled by 2^-e with e chosen from its max |x| so that
// max |x| * 2^-e lies in [2^13, 2^14): nothing overflows and every value within
// 2^-27 of the max stays normal.  The exponents (q, k, v, dO, and dS from the
// bound |dS| <= 2 d max|dO| max|v|) go to the workspace for the backward kernel.

__device__ __forceinline__ int norm_exp(float amax, int target) {
    if (!(amax > 0.f) || !isfinite(amax)) return 0;
    int E;
    frexpf(amax, &E);            // amax = f * 2^E, f in [0.5, 1)
    return E - 1 - target;       // amax * 2^-e in [2^target, 2^(target+1))
}

struct Fp16Job {
    const uint4* src[4];
    uint4* dst[4];
    int64_t n8[4];     // 8-element units of each tensor (n8 of the launch = the largest)
};

// Block-wide max of each thread's m[t] (all >= 0), then one atomicMax per block
// and tensor on the float bits: a same-address atomic from every warp of a
// full grid would serialise in L2 (about 10 us for the ~10^4 warps of one launch).
template <int NT>
__device__ __forceinline__ void block_amax(const float (&m)[NT], unsigned* __restrict__ amax_bits) {
    __shared__ float part[NT][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float v = m[t];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) part[t][warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < NT) {
        float v = part[threadIdx.x][0];
        for (int w = 1; w < nw; ++w) v = fmaxf(v, part[threadIdx.x][w]);
        atomicMax(amax_bits + threadIdx.x, __float_as_uint(v));
    }
}

// max |x| of NT bf16 tensors of job.n8[t] * 8 elements each (float bits, atomicMax)
template <int NT>
__global__ void __launch_bounds__(256)
amax_kernel(int64_t n8, const __grid_constant__ Fp16Job job, unsigned* __restrict__ amax_bits) {
    float m[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) m[t] = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (i >= job.n8[t]) continue;
            const uint4 x = job.src[t][i];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                m[t] = fmaxf(m[t], fmaxf(fabsf(__bfloat162float(v2.x)), fabsf(__bfloat162float(v2.y))));
            }
        }
    }
    block_amax<NT>(m, amax_bits);
}

// fp16 copies dst[t] = src[t] * 2^-e_t, exact; the exponents go to exps[0..NT).
// With ds_d > 0 (the backward: q, k, v, dO) exps[4] gets the dS exponent from
// the bound |dS| <= 2 d max|dO| max|v|.
template <int NT>
__global__ void __launch_bounds__(256)
fp16_copy_kernel(int64_t n8, int ds_d, const __grid_constant__ Fp16Job job,
                 const unsigned* __restrict__ amax_bits, int* __restrict__ exps) {
    float amax[NT], mul[NT];
    int e[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        amax[t] = __uint_as_float(amax_bits[t]);
        e[t] = norm_exp(amax[t], 13);
        mul[t] = ldexpf(1.f, -e[t]);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int t = 0; t < NT; ++t) exps[t] = e[t];
        if (NT == 4 && ds_d > 0) exps[4] = norm_exp(2.f * (float)ds_d * amax[NT - 1] * amax[NT > 2 ? 2 : 0], 14);
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (i >= job.n8[t]) continue;
            const uint4 x = job.src[t][i];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
                __half2 h2 = __floats2half2_rn(__bfloat162float(v2.x) * mul[t], __bfloat162float(v2.y) * mul[t]);
                r[q] = *reinterpret_cast<uint32_t*>(&h2);
            }
            job.dst[t][i] = make_uint4(r[0], r[1], r[2], r[3]);
        }
    }
}

// max |x| over nrows strided rows of row8 8-element units (bf16), one warp per row
__global__ void __launch_bounds__(256)
amax_rows_kernel(int64_t nrows, int row8, int64_t pitch8, const uint4* __restrict__ src,
                 unsigned* __restrict__ amax_bits) {
    const int lane = threadIdx.x & 31;
    float m = 0.f;
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < nrows;
         r += (int64_t)gridDim.x * (blockDim.x >> 5)) {
        const uint4* row = src + r * pitch8;
        for (int c = lane; c < row8; c += 32) {
            const uint4 x = row[c];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                m = fmaxf(m, fmaxf(fabsf(__bfloat162float(v2.x)), fabsf(__bfloat162float(v2.y))));
            }
        }
    }
    const float mm[1] = {m};
    block_amax<1>(mm, amax_bits);
}

// dst = src * 2^-e over the same strided rows (exact fp16), e -> exps[0]
__global__ void __launch_bounds__(256)
fp16_copy_rows_kernel(int64_t nrows, int row8, int64_t pitch8, const uint4* __restrict__ src,
                      uint4* __restrict__ dst, const unsigned* __restrict__ amax_bits, int* __restrict__ exps) {
    const int e = norm_exp(__uint_as_float(amax_bits[0]), 13);
    const float mul = ldexpf(1.f, -e);
    if (blockIdx.x == 0 && threadIdx.x == 0) exps[0] = e;
    const int lane = threadIdx.x & 31;
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < nrows;
         r += (int64_t)gridDim.x * (blockDim.x >> 5)) {
        const uint4* srow = src + r * pitch8;
        uint4* drow = dst + r * pitch8;
        for (int c = lane; c < row8; c += 32) {
            const uint4 x = srow[c];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w[q]);
                __half2 h2 = __floats2half2_rn(__bfloat162float(v2.x) * mul, __bfloat162float(v2.y) * mul);
                o[q] = *reinterpret_cast<uint32_t*>(&h2);
            }
            drow[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

int fp16_grid(int64_t n8) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    const int64_t want = (n8 + 255) / 256;
    return (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
}

}  // namespace

int launch_fp16_copies(const BwdArgs& a, int64_t S, void* stream, int64_t Skv) {
    if (Skv < 0) Skv = S;
    const int64_t nq8 = (int64_t)a.B * S * a.H * a.d / 8, nkv8 = (int64_t)a.B * Skv * a.H * a.d / 8;
    const int64_t n8 = nq8 > nkv8 ? nq8 : nkv8;
    Fp16Job job;
    const void* src[4] = {a.q, a.k, a.v, a.dout};
    for (int t = 0; t < 4; ++t) {
        job.src[t] = static_cast<const uint4*>(src[t]);
        job.dst[t] = static_cast<uint4*>(a.h16[t]);
        job.n8[t] = (t == 1 || t == 2) ? nkv8 : nq8;   // q, dO: the query rows; k, v: the key rows
    }
    const int grid = fp16_grid(n8);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    amax_kernel<4><<<grid, 256, 0, st>>>(n8, job, a.amax_bits);
    fp16_copy_kernel<4><<<grid, 256, 0, st>>>(n8, a.d, job, a.amax_bits, a.exps);
    return (int)cudaGetLastError();
}

int launch_fp16_copy1(const void* src, void* dst, int64_t elems, unsigned* amax_bits, int* exps,
                      void* stream) {
    const int64_t n8 = elems / 8;
    Fp16Job job{};
    job.src[0] = static_cast<const uint4*>(src);
    job.dst[0] = static_cast<uint4*>(dst);
    job.n8[0] = n8;
    const int grid = fp16_grid(n8);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return (int)e;
    amax_kernel<1><<<grid, 256, 0, st>>>(n8, job, amax_bits);
    fp16_copy_kernel<1><<<grid, 256, 0, st>>>(n8, 0, job, amax_bits, exps);
    return (int)cudaGetLastError();
}

int launch_fp16_copy_rows(const void* src, void* dst, int64_t nrows, int row8, int64_t pitch8,
                          unsigned* amax_bits, int* exps, void* stream) {
    const int grid = fp16_grid(nrows * 32);    // 8 rows (warps) per 256-thread block
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return (int)e;
    amax_rows_kernel<<<grid, 256, 0, st>>>(nrows, row8, pitch8, static_cast<const uint4*>(src), amax_bits);
    fp16_copy_rows_kernel<<<grid, 256, 0, st>>>(nrows, row8, pitch8, static_cast<const uint4*>(src),
                                                static_cast<uint4*>(dst), amax_bits, exps);
    return (int)cudaGetLastError();
}

int launch_dq_convert(const BwdArgs& a, int64_t S, int dtype, void* stream) {
    const int64_t n = (int64_t)a.B * S * a.H * a.d;
    const int grid = grid_for(n / 32 + 1);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == ST_DTYPE_F32)
        convert_kernel<float><<<grid, 256, 0, st>>>(n, a.dq_acc, static_cast<float*>(a.dq));
    else
        convert_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(n, a.dq_acc, static_cast<__nv_bfloat16*>(a.dq));
    return (int)cudaGetLastError();
}

int launch_permute(const SegTable& t, int B, int H, int d, int dtype, int to_natural,
                   const void* in, void* out, void* stream) {
    const int row_bytes = d * (dtype == ST_DTYPE_F32 ? 4 : 2);
    const int64_t rows = (int64_t)B * t.S;
    permute_kernel<<<grid_for(rows), kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        t, B, H, row_bytes, to_natural, static_cast<const uint4*>(in), static_cast<uint4*>(out));
    return (int)cudaGetLastError();
}

}  // namespace st
