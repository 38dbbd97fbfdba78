// Group normalisation of a row-sharded image (sm_103a).
//
// ShardTensor summary, "ShardTensor" section 2, implementation details,
// communication: normalisation over a spatially sharded input needs a
// collective (an all-reduce of statistics) to give the numbers of the layer on
// the whole input.  Channels last: shard r is x_r [L_r, W, C] bf16; C splits
// into G groups of C/G channels; group g is normalised with the mean and the
// biased variance of all its values over every shard:
//   y[i, j, c] = (x[i, j, c] - mu_g) / sqrt(var_g + eps) * gamma[c] + beta[c].
//
// Three launches, all HBM-bound:
//   gn_stats_kernel    each block: per group, the count, mean and squared
//                      deviations (M2) of the values it reads (every thread
//                      keeps sums shifted by its first value, in fp32, then
//                      the block merges its threads by the pairwise rule);
//   gn_combine_kernel  the all-reduce: one block per group adds up the blocks'
//                      statistics as fp64 sums -> mean, 1/std;
//   gn_apply_kernel    y = (x - mean) * (gamma / std) + beta, bf16 or fp32,
//                      walked in the opposite order to the statistics pass so
//                      that the rows read last there are still in L2.
// Every thread handles 16-byte vectors (8 channels of one pixel).  Because
// the vectors of one pixel (C / 8 of them) divide the 256 threads of a block,
// a thread's vectors always hold the same 8 channels, so its group, gamma
// and beta are fixed.
#include <cuda_bf16.h>

#include "common.h"

namespace st {
namespace {

constexpr int kGnShards = ST_CONV_MAX_SHARDS;
constexpr int kGnThreads = 256;

struct GnParams {
    const void* in[kGnShards];     // [L_r, W, C] bf16
    void* out[kGnShards];          // [L_r + 2*out_pad, W, C]
    int64_t pix_off[kGnShards + 1];  // first pixel of each shard in the stacked image
    int D, W, C, G, out_pad, out_f32;
    int vshift;                    // log2(C / 8): 16-byte vectors per pixel
    float eps;
    const float* gamma;            // [C] or null (1)
    const float* beta;             // [C] or null (0)
    float* partial;                // [nblocks][G][3]: count, mean, M2
    double* stats;                 // [G][2]: mean, 1/std
    int nblocks;
};

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// (n, mean, M2) of a and b combined (Chan, Golub, LeVeque)
template <typename T>
__device__ __forceinline__ void merge(T& n, T& mean, T& m2, T nb, T meanb, T m2b) {
    if (nb == T(0)) return;
    const T nn = n + nb;
    const T delta = meanb - mean;
    mean += delta * (nb / nn);
    m2 += m2b + delta * delta * (n * nb / nn);
    n = nn;
}

__global__ void __launch_bounds__(kGnThreads) gn_stats_kernel(const __grid_constant__ GnParams p) {
    __shared__ float sn[kGnThreads], smean[kGnThreads], sm2[kGnThreads];
    const int vpp = 1 << p.vshift;                 // vectors per pixel; divides kGnThreads
    const int64_t total = p.pix_off[p.D] << p.vshift;
    const int64_t stride = (int64_t)gridDim.x * kGnThreads;
    const int lane = threadIdx.x & (vpp - 1);      // the same 8 channels in every vector of this thread
    int r = 0;
    float shift = 0.f, s1 = 0.f, s2 = 0.f;
    float cnt = 0.f;
    auto load = [&](int64_t idx) {
        const int64_t pix = idx >> p.vshift;
        while (pix >= p.pix_off[r + 1]) ++r;
        // a plain load: the rows read last stay in L2 for the apply pass
        return static_cast<const uint4*>(p.in[r])[((pix - p.pix_off[r]) << p.vshift) + lane];
    };
    auto add = [&](const uint4 v) {
        float f[8];
        unpack8(v, f);
        if (cnt == 0.f) shift = f[0];
        float a1 = 0.f, a2 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float d = f[i] - shift;
            a1 += d;
            a2 = fmaf(d, d, a2);
        }
        s1 += a1;
        s2 += a2;
        cnt += 8.f;
    };
    int64_t idx = (int64_t)blockIdx.x * kGnThreads + threadIdx.x;
    // four loads in flight per thread
    for (; idx + 3 * stride < total; idx += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = load(idx + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) add(v[u]);
    }
    for (; idx < total; idx += stride) add(load(idx));
    const float mean = cnt > 0.f ? shift + s1 / cnt : 0.f;
    sn[threadIdx.x] = cnt;
    smean[threadIdx.x] = mean;
    sm2[threadIdx.x] = cnt > 0.f ? fmaxf(s2 - s1 * (s1 / cnt), 0.f) : 0.f;
    __syncthreads();
    // thread g merges the threads that read group g: lanes (g*cg/8 .. +cg/8) of
    // every pixel slot of the block
    const int lanes = (p.C / p.G) / 8;
    for (int g = threadIdx.x; g < p.G; g += kGnThreads) {
        float n = 0.f, m = 0.f, q = 0.f;
        for (int t = g * lanes; t < kGnThreads; t += vpp)
            for (int l = 0; l < lanes; ++l) merge(n, m, q, sn[t + l], smean[t + l], sm2[t + l]);
        float* dst = p.partial + ((int64_t)blockIdx.x * p.G + g) * 3;
        dst[0] = n;
        dst[1] = m;
        dst[2] = q;
    }
}

// one block per group: the all-reduce of the blocks' statistics.  In fp64
// the pairwise rule needs a division per merge, which is slow; plain sums of
// n, n*mean and M2 + n*mean^2 need none, and the one subtraction left at the
// end (E[x^2] - mean^2) loses nothing that matters in 53 bits unless the mean
// is beyond about 1e5 standard deviations.
__global__ void __launch_bounds__(kGnThreads) gn_combine_kernel(const __grid_constant__ GnParams p) {
    __shared__ double sn[kGnThreads], s1[kGnThreads], s2[kGnThreads];
    const int g = blockIdx.x;
    double n = 0.0, a = 0.0, q = 0.0;
    for (int b = threadIdx.x; b < p.nblocks; b += kGnThreads) {
        const float* src = p.partial + ((int64_t)b * p.G + g) * 3;
        const double nb = src[0], mb = src[1];
        n += nb;
        a += nb * mb;
        q += (double)src[2] + nb * mb * mb;
    }
    sn[threadIdx.x] = n;
    s1[threadIdx.x] = a;
    s2[threadIdx.x] = q;
    __syncthreads();
    for (int h = kGnThreads / 2; h > 0; h >>= 1) {
        if (threadIdx.x < h) {
            sn[threadIdx.x] += sn[threadIdx.x + h];
            s1[threadIdx.x] += s1[threadIdx.x + h];
            s2[threadIdx.x] += s2[threadIdx.x + h];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double mean = sn[0] > 0.0 ? s1[0] / sn[0] : 0.0;
        const double var = sn[0] > 0.0 ? fmax(s2[0] / sn[0] - mean * mean, 0.0) : 0.0;
        p.stats[2 * g] = mean;
        p.stats[2 * g + 1] = 1.0 / sqrt(var + (double)p.eps);
    }
}

__device__ __forceinline__ uint32_t pack_bf16_pair(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kGnThreads, 4) gn_apply_kernel(const __grid_constant__ GnParams p) {
    const int vpp = 1 << p.vshift;
    const int64_t total = p.pix_off[p.D] << p.vshift;
    const int64_t stride = (int64_t)gridDim.x * kGnThreads;
    // this thread's 8 channels (fixed: the stride is a multiple of vpp)
    const int64_t first = (int64_t)blockIdx.x * kGnThreads + threadIdx.x;
    const int lane = threadIdx.x & (vpp - 1);
    const int c0 = lane * 8;
    const int g = c0 / (p.C / p.G);
    const float mean = (float)p.stats[2 * g];
    const float rstd = (float)p.stats[2 * g + 1];
    float a[8], b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        a[i] = rstd * (p.gamma ? p.gamma[c0 + i] : 1.f);
        b[i] = p.beta ? p.beta[c0 + i] : 0.f;
    }
    int r = p.D - 1;
    auto locate = [&](int64_t idx, int64_t& lp) {
        const int64_t pix = idx >> p.vshift;
        while (pix < p.pix_off[r]) --r;
        lp = pix - p.pix_off[r];
        return r;
    };
    auto store = [&](int rr, int64_t lp, const uint4 v) {
        float f[8];
        unpack8(v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = fmaf(f[i] - mean, a[i], b[i]);
        const int64_t o = ((int64_t)p.out_pad * p.W + lp) * p.C + c0;   // element offset in the padded output
        if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out[rr]) + o);
            __stcs(dst, make_float4(f[0], f[1], f[2], f[3]));
            __stcs(dst + 1, make_float4(f[4], f[5], f[6], f[7]));
        } else {
            __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out[rr]) + o),
                   make_uint4(pack_bf16_pair(f[0], f[1]), pack_bf16_pair(f[2], f[3]), pack_bf16_pair(f[4], f[5]),
                              pack_bf16_pair(f[6], f[7])));
        }
    };
    // backwards through the same vectors the statistics pass visited forwards,
    // four loads in flight per thread
    int64_t s = first < total ? (total - 1 - first) / stride : -1;
    for (; s >= 3; s -= 4) {
        uint4 v[4];
        int rr[4];
        int64_t lp[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            rr[u] = locate(first + (s - u) * stride, lp[u]);
            v[u] = static_cast<const uint4*>(p.in[rr[u]])[(lp[u] << p.vshift) + lane];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) store(rr[u], lp[u], v[u]);
    }
    for (; s >= 0; --s) {
        int64_t lp;
        const int rr = locate(first + s * stride, lp);
        store(rr, lp, static_cast<const uint4*>(p.in[rr])[(lp << p.vshift) + lane]);
    }
}

int sm_count() {
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

size_t group_norm_workspace_bytes(int G) {
    return ((size_t)kGnStatBlocks * G * 3 * sizeof(float) + 255) / 256 * 256 + (size_t)G * 2 * sizeof(double);
}

int launch_group_norm(int D, const int64_t* rows, int W, int C, int G, float eps, const void* const* in,
                      const float* gamma, const float* beta, void* const* out, int out_pad, int out_dtype,
                      void* workspace, void* stream) {
    GnParams p;
    p.pix_off[0] = 0;
    for (int r = 0; r < D; ++r) {
        p.in[r] = in[r];
        p.out[r] = out[r];
        p.pix_off[r + 1] = p.pix_off[r] + rows[r] * W;
    }
    for (int r = D; r < kGnShards; ++r) {
        p.in[r] = nullptr;
        p.out[r] = nullptr;
        p.pix_off[r + 1] = p.pix_off[D];
    }
    p.D = D;
    p.W = W;
    p.C = C;
    p.G = G;
    p.out_pad = out_pad;
    p.out_f32 = out_dtype == ST_DTYPE_F32 ? 1 : 0;
    p.vshift = 0;
    while ((8 << p.vshift) < C) ++p.vshift;
    p.eps = eps;
    p.gamma = gamma;
    p.beta = beta;
    p.partial = static_cast<float*>(workspace);
    p.stats = reinterpret_cast<double*>(static_cast<char*>(workspace) +
                                        ((size_t)kGnStatBlocks * G * 3 * sizeof(float) + 255) / 256 * 256);
    // grid-stride kernels: as many blocks as are resident at once (one wave)
    const int64_t vecs = p.pix_off[D] << p.vshift;
    const int64_t want = (vecs + kGnThreads - 1) / kGnThreads;
    auto wave = [&](const void* fn) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kGnThreads, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        int64_t n = (int64_t)sm_count() * per_sm;
        if (n > kGnStatBlocks) n = kGnStatBlocks;
        return (int)(want < n ? want : n);
    };
    p.nblocks = wave(reinterpret_cast<const void*>(gn_stats_kernel));
    const int apply_blocks = wave(reinterpret_cast<const void*>(gn_apply_kernel));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    gn_stats_kernel<<<p.nblocks, kGnThreads, 0, s>>>(p);
    gn_combine_kernel<<<G, kGnThreads, 0, s>>>(p);
    gn_apply_kernel<<<apply_blocks, kGnThreads, 0, s>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace st
