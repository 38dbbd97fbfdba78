// fp32 SIMT attention kernels (forward and backward).
//
// These carry the fp32 path, whose tolerance (max abs 1e-5 against the float64
// definition) rules out tf32 tensor cores: the forward is fp32 FFMA/FADD with
// expf; the backward forms its scores and gradient sums in double (see there).  The structure is the same
// ring walk as the tensor-core path: one CTA per (query tile, b, h), KV shards
// visited in ring order, each KV tile folded into a running (max, sum, O)
// state -- the online form of the log-sum-exp merge of per-shard partials.
#include <cfloat>
#include <type_traits>
#include <cmath>

#include "device.cuh"

namespace st {
namespace {

constexpr int kBM = 64;     // query rows per CTA
constexpr int kBN = 64;     // keys per KV tile
constexpr int kThreads = 256;

__device__ __forceinline__ int64_t row_off(int b, int row, int h, int S, int H, int d) {
    return (((int64_t)b * S + row) * H + h) * (int64_t)d;
}

template <int D>
constexpr int fwd_smem_floats() {
    return 2 * D * (kBM + 4) + kBN * (D + 4) + kBM * (kBN + 4) + 3 * kBM;
}

// Forward.  Thread (ty, tx) = (tid / 16, tid % 16) owns score rows ty*4..+3 x
// key columns tx*4..+3 and output rows ty*4..+3 x columns {tx*4..+3, +64 ..}.
// Softmax: four threads per row, sixteen columns each.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const __grid_constant__ SegTable tab, const __grid_constant__ AttnArgs a) {
    constexpr int LDT = kBM + 4, LDV = D + 4, LDP = kBN + 4, NG = D / 64;
    extern __shared__ float4 smem4[];
    float* Qt = reinterpret_cast<float*>(smem4);   // [D][LDT] transposed Q
    float* Kt = Qt + D * LDT;                      // [D][LDT] transposed K
    float* Vs = Kt + D * LDT;                      // [kBN][LDV]
    float* Ps = Vs + kBN * LDV;                    // [kBM][LDP]
    float* alpha_s = Ps + kBM * LDP;               // [kBM]
    float* m_s = alpha_s + kBM;
    float* l_s = m_s + kBM;

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int H = a.H, S = tab.S;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const QTile qt = locate_qtile(tab, blockIdx.x, kBM);
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);

    for (int e = tid; e < kBM * D; e += kThreads) {
        const int r = e / D, c = e % D;
        Qt[c * LDT + r] = r < qt.nq ? to_f32(q[row_off(b, qt.row0 + r, h, S, H, D) + c]) : 0.f;
    }

    float O[4][4 * NG];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4 * NG; ++c) O[i][c] = 0.f;
    const int srow = tid >> 2, spart = tid & 3;
    float m_run = -INFINITY, l_run = 0.f;
    const float scale = a.scale;

    auto flush = [&](float* dst_out, int64_t out_shard_off, float* dst_lse, int64_t lse_shard_off,
                     bool to_partial) {
        __syncthreads();
        if (spart == 0) {
            m_s[srow] = m_run;
            l_s[srow] = l_run;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= qt.nq) continue;
            const float l = l_s[r];
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t base = row_off(b, qt.row0 + r, h, S, H, D);
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int c = g * 64 + tx * 4 + jj;
                    const float val = O[i][g * 4 + jj] * inv;
                    if (to_partial)
                        dst_out[out_shard_off + base + c] = val;
                    else
                        static_cast<T*>(a.out)[base + c] = from_f32<T>(val);
                }
        }
        if (spart == 0 && srow < qt.nq) {
            const float l = l_run;
            dst_lse[lse_shard_off + ((int64_t)b * H + h) * S + qt.row0 + srow] =
                l > 0.f ? m_run + logf(l) : -INFINITY;
        }
    };

    ring_walk<kBN>(tab, qt.shard, [&](int j, int kv0, int nk, int natk, bool last) {
        const int kind = classify(a.causal, qt.nat0, qt.nq, natk, nk, kBN);
        if (kind != kSkip) {
            __syncthreads();
            for (int e = tid; e < kBN * D; e += kThreads) {
                const int r = e / D, c = e % D;
                float kx = 0.f, vx = 0.f;
                if (r < nk) {
                    const int64_t o = row_off(b, kv0 + r, h, S, H, D) + c;
                    kx = to_f32(k[o]);
                    vx = to_f32(v[o]);
                }
                Kt[c * LDT + r] = kx;
                Vs[r * LDV + c] = vx;
            }
            __syncthreads();
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                const float4 qa = *reinterpret_cast<const float4*>(&Qt[c * LDT + ty * 4]);
                const float4 kb = *reinterpret_cast<const float4*>(&Kt[c * LDT + tx * 4]);
                const float qv[4] = {qa.x, qa.y, qa.z, qa.w};
                const float kv[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(qv[i], kv[jj], acc[i][jj]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int r = ty * 4 + i, c = tx * 4 + jj;
                    bool ok = true;
                    if (kind == kPartial)
                        ok = c < nk && (!a.causal || natk + c <= qt.nat0 + r);
                    Ps[r * LDP + c] = ok ? acc[i][jj] * scale : -INFINITY;
                }
            __syncthreads();
            {
                float* prow = Ps + srow * LDP + spart * 16;
                float mx = -INFINITY;
#pragma unroll
                for (int c = 0; c < 16; ++c) mx = fmaxf(mx, prow[c]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run, mx);
                const float m_ref = m_new == -INFINITY ? 0.f : m_new;
                float sum = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float p = expf(prow[c] - m_ref);
                    prow[c] = p;
                    sum += p;
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                const float al = expf(m_run - m_ref);
                l_run = l_run * al + sum;
                m_run = m_new;
                if (spart == 0) alpha_s[srow] = al;
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float al = alpha_s[ty * 4 + i];
#pragma unroll
                for (int c = 0; c < 4 * NG; ++c) O[i][c] *= al;
            }
#pragma unroll 4
            for (int n = 0; n < kBN; ++n) {
                float vv[4 * NG];
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float4 x = *reinterpret_cast<const float4*>(&Vs[n * LDV + g * 64 + tx * 4]);
                    vv[g * 4 + 0] = x.x;
                    vv[g * 4 + 1] = x.y;
                    vv[g * 4 + 2] = x.z;
                    vv[g * 4 + 3] = x.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float p = Ps[(ty * 4 + i) * LDP + n];
#pragma unroll
                    for (int c = 0; c < 4 * NG; ++c) O[i][c] = fmaf(p, vv[c], O[i][c]);
                }
            }
        }
        if (a.part_out != nullptr && last) {
            const int64_t elems = (int64_t)a.B * S * H * D;
            const int64_t rows = (int64_t)a.B * H * S;
            flush(a.part_out, j * elems, a.part_lse, j * rows, true);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 4 * NG; ++c) O[i][c] = 0.f;
            m_run = -INFINITY;
            l_run = 0.f;
        }
    });
    if (a.part_out == nullptr) flush(nullptr, 0, a.lse, 0, false);
}

// Backward, KV-stationary.  One CTA per (KV tile, b, h) accumulates dK and dV
// for its keys over every query tile and adds its share of dQ into the fp32
// accumulator with atomics.  Thread (ty, tx) owns rows ty + 16 i and columns
// tx + 16 jj of each product (strided, so shared-memory reads do not conflict).
//
// Acc is double for fp32 inputs: every gradient element is a long sum of
// P-weighted terms that cancel (rows of dS sum to zero), and fp32 rounding of
// the scores and of those sums alone comes close to the 1e-5 bound on
// max|error| / RMS.  For bf16 inputs Acc is float.
template <typename T>
using BwdAcc = typename std::conditional<std::is_same<T, float>::value, double, float>::type;

template <typename T, int D>
constexpr size_t bwd_smem_bytes() {
    return sizeof(float) * 4 * kBM * (D + 1) + sizeof(BwdAcc<T>) * (2 * kBM * (kBN + 1) + 2 * kBM);
}

template <typename T, typename TG, int D>
__global__ void __launch_bounds__(kThreads)
bwd_simt_kernel(const __grid_constant__ SegTable tab, const __grid_constant__ BwdArgs a) {
    using Acc = BwdAcc<T>;
    constexpr int LD = D + 1, LP = kBN + 1, NC = D / 16;
    extern __shared__ float4 smem4[];
    Acc* Ps = reinterpret_cast<Acc*>(smem4);
    Acc* dSs = Ps + kBM * LP;
    Acc* lse_s = dSs + kBM * LP;
    Acc* del_s = lse_s + kBM;
    float* Ks = reinterpret_cast<float*>(del_s + kBM);
    float* Vs = Ks + kBN * LD;
    float* Qs = Vs + kBN * LD;
    float* dOs = Qs + kBM * LD;

    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int H = a.H, S = tab.S;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const QTile kt = locate_qtile(tab, blockIdx.x, kBN);   // this CTA's key tile
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* v = static_cast<const T*>(a.v);
    const T* dout = static_cast<const T*>(a.dout);
    const Acc scale = (Acc)a.scale;

    for (int e = tid; e < kBN * D; e += kThreads) {
        const int r = e / D, c = e % D;
        float kx = 0.f, vx = 0.f;
        if (r < kt.nq) {
            const int64_t o = row_off(b, kt.row0 + r, h, S, H, D) + c;
            kx = to_f32(k[o]);
            vx = to_f32(v[o]);
        }
        Ks[r * LD + c] = kx;
        Vs[r * LD + c] = vx;
    }
    Acc dK[4][NC], dV[4][NC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < NC; ++c) dK[i][c] = dV[i][c] = 0;

    for (int qi = 0; qi < tab.ntiles; ++qi) {
        const QTile qt = locate_qtile(tab, qi, kBM);
        const int kind = classify(a.causal, qt.nat0, qt.nq, kt.nat0, kt.nq, kBN);
        if (kind == kSkip) continue;
        __syncthreads();
        for (int e = tid; e < kBM * D; e += kThreads) {
            const int r = e / D, c = e % D;
            float qx = 0.f, dx = 0.f;
            if (r < qt.nq) {
                const int64_t o = row_off(b, qt.row0 + r, h, S, H, D) + c;
                qx = to_f32(q[o]);
                dx = to_f32(dout[o]);
            }
            Qs[r * LD + c] = qx;
            dOs[r * LD + c] = dx;
        }
        if (tid < kBM) {
            const int64_t o = ((int64_t)b * H + h) * S + qt.row0 + tid;
            if constexpr (std::is_same<Acc, double>::value) {
                lse_s[tid] = tid < qt.nq ? a.lse_d[o] : (Acc)INFINITY;
                del_s[tid] = tid < qt.nq ? a.delta_d[o] : (Acc)0;
            } else {
                lse_s[tid] = tid < qt.nq ? a.lse[o] : INFINITY;
                del_s[tid] = tid < qt.nq ? a.delta[o] : 0.f;
            }
        }
        __syncthreads();
        // P and dS for query rows ty + 16 i, key columns tx + 16 jj.
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 16 * i;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int c = tx + 16 * jj;
                Acc s = 0, dp = 0;
#pragma unroll 8
                for (int e = 0; e < D; ++e) {
                    s += (Acc)Qs[r * LD + e] * (Acc)Ks[c * LD + e];
                    dp += (Acc)dOs[r * LD + e] * (Acc)Vs[c * LD + e];
                }
                bool ok = r < qt.nq && c < kt.nq;
                if (a.causal) ok = ok && (kt.nat0 + c <= qt.nat0 + r);
                const Acc p = ok ? exp(s * scale - lse_s[r]) : (Acc)0;
                Ps[r * LP + c] = p;
                dSs[r * LP + c] = p * (dp - del_s[r]);
            }
        }
        __syncthreads();
        // dV += P^T dO ; dK += scale dS^T Q  (key rows ty + 16 i, columns tx + 16 jj)
#pragma unroll 4
        for (int r = 0; r < kBM; ++r) {
            Acc dov[NC], qv[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                dov[c] = dOs[r * LD + tx + 16 * c];
                qv[c] = Qs[r * LD + tx + 16 * c];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const Acc p = Ps[r * LP + ty + 16 * i];
                const Acc ds = dSs[r * LP + ty + 16 * i] * scale;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    dV[i][c] += p * dov[c];
                    dK[i][c] += ds * qv[c];
                }
            }
        }
        // dQ += scale dS K  (query rows ty + 16 i)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty + 16 * i;
            Acc acc[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[c] = 0;
            for (int n = 0; n < kBN; ++n) {
                const Acc ds = dSs[r * LP + n];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[c] += ds * (Acc)Ks[n * LD + tx + 16 * c];
            }
            if (r < qt.nq) {
                float* dst = a.dq_acc + row_off(b, qt.row0 + r, h, S, H, D);
#pragma unroll
                for (int c = 0; c < NC; ++c) atomicAdd(dst + tx + 16 * c, (float)(acc[c] * scale));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 16 * i;
        if (r >= kt.nq) continue;
        const int64_t o = row_off(b, kt.row0 + r, h, S, H, D);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            static_cast<TG*>(a.dk)[o + tx + 16 * c] = from_f32<TG>((float)dK[i][c]);
            static_cast<TG*>(a.dv)[o + tx + 16 * c] = from_f32<TG>((float)dV[i][c]);
        }
    }
}

// Row statistics of the fp32 backward in double: lse_i = log sum_j e^{s_ij}
// and Delta_i = sum_j P_ij dP_ij over the visible keys of row i -- the same
// Delta as rowsum(dO o out) with out = sum_j P_ij v_j, formed without the
// rounding of the stored fp32 out and lse.  In rows with few visible keys
// dP - Delta cancels heavily, and fp32 statistics alone would cost ~1e-5 of
// the gradient's RMS.  One warp per row; lanes stride over the keys.
template <int D>
__global__ void __launch_bounds__(128)
rowstats_f64_kernel(const __grid_constant__ SegTable tab, const __grid_constant__ BwdArgs a) {
    __shared__ double qs[4][D];
    __shared__ double gs[4][D];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, S = tab.S;
    const int64_t rid = (int64_t)blockIdx.x * 4 + w;
    if (rid >= (int64_t)a.B * H * S) return;
    const int t = (int)(rid % S);
    const int bh = (int)(rid / S);
    const int b = bh / H, h = bh % H;
    const float* q = static_cast<const float*>(a.q);
    const float* k = static_cast<const float*>(a.k);
    const float* v = static_cast<const float*>(a.v);
    const float* g = static_cast<const float*>(a.dout);
    for (int c = lane; c < D; c += 32) {
        qs[w][c] = q[row_off(b, t, h, S, H, D) + c];
        gs[w][c] = g[row_off(b, t, h, S, H, D) + c];
    }
    __syncwarp();
    int st = 0;
    while (st + 1 < tab.nseg && tab.seg_buf[st + 1] <= t) ++st;
    const int pos_t = tab.seg_nat[st] + (t - tab.seg_buf[st]);
    const double scale = (double)a.scale;
    double m = -INFINITY, l = 0.0;
    for (int s = 0; s < tab.nseg; ++s) {
        for (int j = tab.seg_buf[s] + lane; j < tab.seg_buf[s + 1]; j += 32) {
            if (a.causal && tab.seg_nat[s] + (j - tab.seg_buf[s]) > pos_t) continue;
            const float* kr = k + row_off(b, j, h, S, H, D);
            double dot = 0.0;
            for (int c = 0; c < D; ++c) dot += qs[w][c] * (double)kr[c];
            const double x = dot * scale;
            if (x > m) {
                l = l * exp(m - x) + 1.0;
                m = x;
            } else {
                l += exp(x - m);
            }
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        const double m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const double l2 = __shfl_xor_sync(0xffffffffu, l, off);
        const double mm = fmax(m, m2);
        if (mm != -INFINITY) {
            l = (m == -INFINITY ? 0.0 : l * exp(m - mm)) + (m2 == -INFINITY ? 0.0 : l2 * exp(m2 - mm));
            m = mm;
        }
    }
    const double lse = m + log(l);
    double dl = 0.0;
    for (int s = 0; s < tab.nseg; ++s) {
        for (int j = tab.seg_buf[s] + lane; j < tab.seg_buf[s + 1]; j += 32) {
            if (a.causal && tab.seg_nat[s] + (j - tab.seg_buf[s]) > pos_t) continue;
            const float* kr = k + row_off(b, j, h, S, H, D);
            const float* vr = v + row_off(b, j, h, S, H, D);
            double dot = 0.0, dp = 0.0;
            for (int c = 0; c < D; ++c) {
                dot += qs[w][c] * (double)kr[c];
                dp += gs[w][c] * (double)vr[c];
            }
            dl += exp(dot * scale - lse) * dp;
        }
    }
    for (int off = 16; off > 0; off >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, off);
    if (lane == 0) {
        const int64_t o = ((int64_t)b * H + h) * S + t;
        a.lse_d[o] = lse;
        a.delta_d[o] = dl;
    }
}

template <typename T, int D>
int launch_fwd_simt_t(const SegTable& t, const AttnArgs& a, void* stream) {
    const size_t smem = sizeof(float) * fwd_smem_floats<D>();
    auto kern = fwd_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(t.ntiles, a.B * a.H);
    kern<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(t, a);
    return (int)cudaGetLastError();
}

template <typename T, typename TG, int D>
int launch_bwd_simt_t(const SegTable& t, const BwdArgs& a, void* stream) {
    const size_t smem = bwd_smem_bytes<T, D>();
    auto kern = bwd_simt_kernel<T, TG, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(t.ntiles, a.B * a.H);
    kern<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(t, a);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_fwd_simt(const SegTable& t, const AttnArgs& a, int dtype, void* stream) {
    if (dtype == ST_DTYPE_F32)
        return a.d == 64 ? launch_fwd_simt_t<float, 64>(t, a, stream)
                         : launch_fwd_simt_t<float, 128>(t, a, stream);
    return a.d == 64 ? launch_fwd_simt_t<__nv_bfloat16, 64>(t, a, stream)
                     : launch_fwd_simt_t<__nv_bfloat16, 128>(t, a, stream);
}

int launch_rowstats_f64(const SegTable& t, const BwdArgs& a, void* stream) {
    const int64_t rows = (int64_t)a.B * a.H * t.S;
    const int grid = (int)((rows + 3) / 4);
    if (a.d == 64)
        rowstats_f64_kernel<64><<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(t, a);
    else
        rowstats_f64_kernel<128><<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(t, a);
    return (int)cudaGetLastError();
}

int launch_bwd_simt(const SegTable& t, const BwdArgs& a, int dtype, void* stream) {
    // fp32 inputs only: bf16 runs on the tensor-core backward
    if (dtype != ST_DTYPE_F32) return (int)cudaErrorInvalidValue;
    return a.d == 64 ? launch_bwd_simt_t<float, float, 64>(t, a, stream)
                     : launch_bwd_simt_t<float, float, 128>(t, a, stream);
}

}  // namespace st
