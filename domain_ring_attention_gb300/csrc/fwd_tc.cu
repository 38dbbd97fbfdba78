// Forward sharded ring attention on tcgen05 tensor cores (sm_103a), bf16 in,
// fp32 accumulation, bf16 out + fp32 lse.
//
// One CTA owns 256 query rows (two 128-row halves of one segment) of one
// (batch, head) and walks the KV tiles in ring order: KV shard r, r-1, ...,
// r+1 (mod D) for a query tile of shard r, the order in which rank r of a ring
// receives its neighbours' K/V (ShardTensor summary, section 4, ring
// attention).  On one GPU every shard is a row range of the same HBM buffer,
// so "receiving" a shard is a TMA load of its next 128-key tile.  The running
// (max, sum, O) state carried from tile to tile and shard to shard is the
// log-sum-exp merge of the per-shard partials, done incrementally.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: Q (d = 128) once, then K and V tiles into a
//                smem ring.
//   warp 1       TMEM allocator and single-thread MMA issuer:
//                  S_t = Q_t K^T    (tcgen05.mma; Q from TMEM at d = 64, else smem)
//                  O_t += P_t V     (tcgen05.mma, A = P from TMEM, B from smem)
//   warps 4-7    softmax for query half 0, warps 8-11 for half 1: read S_t from
//                TMEM, mask (shard tails, causal / zigzag order), online
//                softmax in the log2 domain, write P_t (fp16) back over S_t,
//                rescale O_t when the running max grows by more than 2^8, and
//                finally normalise O_t and store out / lse.
// Tensor memory: S_0 | S_1 | O_0 | O_1 (128 + 128 + D + D of 512 columns; at
// d = 64 each O carries 16 more columns, the first of which accumulates the
// row sums of P through a column of ones beside V).
// S = Q K^T runs on the bf16 inputs.  O += P V runs in fp16: P (<= 2^8 with the
// stale-max rescaling) keeps 11 significant bits instead of bf16's 8, and V is
// an exact fp16 copy scaled by a power of two (made before the launch).  The
// output error is then ~8x below that of a bf16 P, which also matters for
// the backward's Delta = rowsum(dO o out).
// Every barrier wait is bounded (see tc_ptx.cuh).
#include <cuda.h>
#include <cuda_fp16.h>

#include <cmath>
#include <algorithm>
#include <type_traits>
#include <mutex>
#include <vector>

#include "device.cuh"
#include "tc_ptx.cuh"

namespace st {
namespace {

using namespace tc;

constexpr int kM = 128;          // rows per query half (MMA M)
constexpr int kNQ = 2;           // query halves per CTA
constexpr int kN = 128;          // keys per KV tile
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;   // rescale O only when the max grows by > 2^8
constexpr int kMaxOrder = 4096;        // longest tile order passed as a kernel parameter

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms per row
    static constexpr int kChunkBytes = kM * 128;           // 128 rows x 64 bf16
    static constexpr int kTileBytes = kChunks * kChunkBytes;
    static constexpr int kStages = D == 64 ? 4 : 2;
    // d = 64: the row sums of P come out of the P V product itself.  Each V
    // stage carries a second 64-column swizzle atom (at the descriptor's
    // leading byte offset) whose column 0 is all ones, the MMA runs with
    // N = 80, and O's column 64 accumulates sum_j P_ij -- the sum of exactly
    // the fp16 P values that weight V -- with no per-score add in the softmax.
    // (d = 128 has no TMEM left for the extra 2 x 16 columns.)
    static constexpr bool kSumCol = D == 64;
    // d = 64: PV_t in two halves of 64 keys, the first issued as soon as the
    // softmax has written P for them (at d = 128 the extra live registers of
    // the early rescale cost more than the earlier PV saves)
    static constexpr bool kHalfP = D == 64;
    static constexpr int kOCols = D + (kSumCol ? 16 : 0);
    static constexpr int kVStageBytes = kTileBytes + (kSumCol ? kChunkBytes : 0);
    // d = 64: Q is kept in tensor memory as the A operand of S = Q K^T, so
    // the S MMAs read only K from shared memory (an SS MMA of N = 128 reads
    // 8 KB of shared memory per K step, close to the 128 B/clk the SM's
    // shared memory delivers while the tensor core needs ~73 clocks for it).
    static constexpr bool kQTmem = D == 64;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + (kQTmem ? 0 : kNQ * kTileBytes);
    static constexpr int kVOff = kKOff + kStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kStages * kVStageBytes;
    // q_full, kv_full[S], kv_empty[S], s_full[NQ], p_full[NQ], o_done[NQ], drain, p_half[NQ]
    static constexpr int kNumBars = 2 + 2 * kStages + 4 * kNQ;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kNQ * kN + kNQ * kOCols + (kQTmem ? kNQ * D / 2 : 0) <= (int)kTmemCols,
                  "tensor memory columns");
    __host__ __device__ static constexpr uint32_t s_col(int t) { return (uint32_t)(t * kN); }
    __host__ __device__ static constexpr uint32_t o_col(int t) { return (uint32_t)(kNQ * kN + t * kOCols); }
    // Q_t as bf16 pairs: column c holds elements 2c and 2c + 1 of the row
    __host__ __device__ static constexpr uint32_t q_col(int t) {
        return (uint32_t)(kNQ * kN + kNQ * kOCols + t * (D / 2));
    }
};

struct FwdParams {
    CUtensorMap tq;
    CUtensorMap tk;
    CUtensorMap tv;
    SegTable tab;              // query tiles of kNQ * kM rows (q, out, lse)
    SegTable kvtab;            // the keys (k, v): the same layout, or in a ring step another shard
    const void* q;             // bf16 [B,S,H,D] (read directly when Q lives in TMEM)
    void* out;                 // bf16, or fp32 when out_f32
    float* lse;
    int B, H;
    float scale_log2;          // softmax scale * log2(e)
    int causal;
    int out_f32;
    const int* exps;           // exps[0]: v16 = v * 2^-exps[0]
    // partials mode: per-KV-shard (O_j normalised, lse_j), [D,B,S,H,d] / [D,B,H,S]
    float* part_out;
    float* part_lse;
    // ring step: running state (fp32 out and lse of the query rows) that this
    // launch's result is merged into by the log-sum-exp rule, or nullptr
    const float* prev_out;
    const float* prev_lse;
    int use_order;             // causal: CTAs take tiles heaviest first
    int tile0;                 // first query tile of this launch (without an order)
    uint16_t order[kMaxOrder];
};

// The parameters of a launch over the heads h0 .. h0 + hn - 1 only (grid y = B * hn):
// the host-buffer forward computes the heads in groups.  A type of its own, so
// that the ordinary launches keep their parameter block as it is.
struct FwdParamsHeads : FwdParams {
    int h0, hn;
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// The softmax pass of a tile on the causal diagonal, one row per lane: P =
// 2^(S * sl2 - m_ref) split into fp16 hi and lo parts (P = P_hi + P_lo, P_hi
// over S's columns 0-63, P_lo over columns 64-127; keys past `limit` masked).
// Returns the row's sum of P over the tile (kSum).  Not inlined: inlined into
// the softmax loop, the registers of the two parts made the compiler spill on
// every tile of the causal kernels, not only on these (the forward ran ~8 %
// slower).  S is read again from tensor memory, columns 64-127 (where P_lo
// goes) first, so that no store of this pass overwrites scores not yet read.
// With kHalfP (d = 64) the keys 0-63 signal goes out halfway, as in the
// ordinary pass; the caller has rescaled O before.
template <bool kSum, bool kHalfP>
__device__ __noinline__ float diag_pass(uint32_t tS, float sl2, float m_ref, int limit, uint32_t bar_half) {
    uint32_t s23[2][32];
    tmem_ld32(tS + 64, s23[0]);
    tmem_ld32(tS + 96, s23[1]);
    tmem_wait_ld();
    const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m_ref, -m_ref);
    uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t s01[32];
        if (c < 2) {
            tmem_ld32(tS + c * 32, s01);
            tmem_wait_ld();
        }
        if (kHalfP && c == 2) {
            // keys 0-63 (hi and lo parts) are written
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(bar_half);
        }
        uint32_t pk[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int k = 32 * c + 2 * i;
            const uint32_t u0 = c < 2 ? s01[2 * i] : s23[c & 1][2 * i];
            const uint32_t u1 = c < 2 ? s01[2 * i + 1] : s23[c & 1][2 * i + 1];
            const float v0 = k > limit ? -INFINITY : __uint_as_float(u0);
            const float v1 = k + 1 > limit ? -INFINITY : __uint_as_float(u1);
            float x0, x1;
            f2_unpack(ffma2(f2_pack(v0, v1), sl2x2, negm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            if constexpr (kSum) {
                if (i & 1)
                    acc1 = fadd2(acc1, f2_pack(p0, p1));
                else
                    acc0 = fadd2(acc0, f2_pack(p0, p1));
            }
            pk[i] = pack_f16(p0, p1);
            const float2 hi = __half22float2(__floats2half2_rn(p0, p1));
            pl[i] = pack_f16(p0 - hi.x, p1 - hi.y);
        }
        tmem_st16(tS + c * 16, pk);
        tmem_st16(tS + 64 + c * 16, pl);
    }
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    if constexpr (kSum) {
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, b0, b1);
    }
    return (a0 + a1) + (b0 + b1);
}

// Kind of the (query half, KV tile) pair; an empty half skips everything.
__device__ __forceinline__ int half_kind(int causal, int nat0, int nq, int natk, int nk) {
    if (nq <= 0) return kSkip;
    return classify(causal, nat0, nq, natk, nk, kN);
}

// kSplit: compiled with the mask and the hi/lo path for partial tiles (causal
// masks or ragged shards; the hi/lo split itself only on the causal diagonal);
// layouts whose tiles are all full use the kernel without either.
// kMode: what the kernel writes.
//   kFused    out, lse of the whole ring (the running state carried across KV shards)
//   kParts    the partials mode -- instead of carrying the running state from one
//             KV shard to the next, the state is normalised and written out at the
//             end of every KV shard (O_j / l_j and lse_j = m_j + ln l_j: what one
//             ring step hands to the merge) and restarted; a shard with no visible
//             key gives O_j = 0 and lse_j = -inf.  Compiled with kSplit.
//   kMerge    a ring step: out, lse of this launch's keys merged by the log-sum-exp
//             rule into the running state prev_out, prev_lse.  Compiled with kSplit.
enum { kFused = 0, kParts = 1, kMerge = 2 };

// kHeads: the launch covers the heads h0 .. h0 + hn - 1 only (FwdParamsHeads);
// a separate instantiation, so that the ordinary launches keep the plain (b, h)
// decoding.
template <int D, bool kSplit, int kMode, bool kHeads>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ std::conditional_t<kHeads, FwdParamsHeads, FwdParams> p) {
    static_assert(kSplit || kMode == kFused, "partials and ring steps walk the ring with the split kernel");
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t sQ = sbase + C::kQOff, sK = sbase + C::kKOff, sV = sbase + C::kVOff;
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t bar_q = bars;
    // K and V of a tile land on one barrier: with the ring several tiles
    // deep, both are there long before S needs K, and the MMA issuer polls
    // one barrier per tile instead of two
    auto bar_kv = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_e = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
    auto bar_s = [&](int t) { return bars + 8u * (1 + 2 * C::kStages + t); };
    auto bar_p = [&](int t) { return bars + 8u * (1 + 2 * C::kStages + kNQ + t); };
    auto bar_o = [&](int t) { return bars + 8u * (1 + 2 * C::kStages + 2 * kNQ + t); };
    const uint32_t bar_drain = bars + 8u * (1 + 2 * C::kStages + 3 * kNQ);
    // P_t of keys 0-63 written (PV_t runs in two halves of 64 keys)
    auto bar_pa = [&](int t) { return bar_drain + 8u * (1 + t); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H;
    int b, h;
    if constexpr (kHeads) {
        b = blockIdx.y / p.hn;
        h = p.h0 + blockIdx.y % p.hn;
    } else {
        b = blockIdx.y / H;
        h = blockIdx.y % H;
    }
    const int tile = p.use_order ? (int)p.order[blockIdx.x] : p.tile0 + (int)blockIdx.x;
    const QTile qt = locate_qtile(p.tab, tile, kNQ * kM);
    int nq_h[kNQ], nat_h[kNQ];
#pragma unroll
    for (int t = 0; t < kNQ; ++t) {
        nq_h[t] = min(kM, max(0, qt.nq - kM * t));
        nat_h[t] = qt.nat0 + kM * t;
    }
    const int causal = p.causal;
    auto active = [&](int nk, int natk) {
        bool any = false;
#pragma unroll
        for (int t = 0; t < kNQ; ++t) any |= half_kind(causal, nat_h[t], nq_h[t], natk, nk) != kSkip;
        return any;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar_q, C::kQTmem ? kNQ * kM / 32 : 1);     // one arrival per softmax warp
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_kv(s), 1);
            mbar_init(bar_e(s), 1);
        }
        for (int t = 0; t < kNQ; ++t) {
            mbar_init(bar_s(t), 1);
            mbar_init(bar_p(t), 4);                          // one arrival per warp of the half
            mbar_init(bar_pa(t), 4);
            mbar_init(bar_o(t), 1);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tq);
        prefetch_tmap(&p.tk);
        prefetch_tmap(&p.tv);
    }
    if constexpr (C::kSumCol) {
        // The ones atom of every V stage, in the 128-byte-swizzled MN-major
        // layout of the V tiles: key row r is 128 bytes at r * 128, and its
        // 16-byte unit u sits at unit position u ^ (r & 7).  Column 0 (unit 0,
        // first half) is 1.0 in fp16, every other column 0.
        if (warp == 2 || warp == 3) {
            const int t = threadIdx.x - 64;                 // 0..63
            for (int s = 0; s < C::kStages; ++s) {
                uint4* atom = reinterpret_cast<uint4*>(gbase + C::kVOff + s * C::kVStageBytes + C::kTileBytes);
                for (int u = t; u < C::kChunkBytes / 16; u += 64) {
                    const int r = u >> 3, pos = u & 7;      // row r, unit position pos
                    atom[u] = make_uint4(pos == (r & 7) ? 0x3C00u : 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async();                            // visible to the tensor core
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            if constexpr (!C::kQTmem) {
                mbar_arrive_expect_tx(bar_q, kNQ * C::kTileBytes);
                for (int t = 0; t < kNQ; ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &p.tq, bar_q, c * 64, h,
                                    qt.row0 + kM * t, b);
            }
            int j = 0;
            bool ok = true;
            ring_walk<kN>(p.kvtab, qt.shard, [&](int, int kv0, int nk, int natk, bool) {
                if (!ok || !active(nk, natk)) return;
                const int s = j % C::kStages;
                if (j >= C::kStages) ok = mbar_wait(bar_e(s), ((j / C::kStages) - 1) & 1, abort_flag);
                if (!ok) return;
                mbar_arrive_expect_tx(bar_kv(s), 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(sK + s * C::kTileBytes + c * C::kChunkBytes, &p.tk, bar_kv(s), c * 64, h,
                                kv0, b);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(sV + s * C::kVStageBytes + c * C::kChunkBytes, &p.tv, bar_kv(s), c * 64, h,
                                kv0, b);
                ++j;
            });
            // Let every load this thread issued land before the CTA can exit
            // (also after an abort: the drain waits ignore the abort word).
            if constexpr (!C::kQTmem) mbar_wait_drain(bar_q, 0);
            for (int jj = max(0, j - C::kStages); jj < j; ++jj) {
                const int s = jj % C::kStages;
                const uint32_t ph = (jj / C::kStages) & 1;
                mbar_wait_drain(bar_kv(s), ph);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // Issue order on the tensor pipe (ping-pong of the two halves):
        //   S0(0) S1(0) | PV0(0) S0(1) PV1(0) S1(1) | PV0(1) S0(2) ...
        // so that while one softmax warpgroup works on S_t, the tensor core
        // runs the other half's PV and next S, and the two warpgroups stay
        // staggered.  S_t(j+1) overwrites P_t(j), which PV_t(j) reads: the
        // tcgen05.mma operations of one thread execute in issue order, so it
        // needs no wait.  The loop is kept lean (descriptors precomputed, a
        // stage or K step adds its byte offset >> 4 to the start-address
        // field): at d = 64 the tensor core runs a tile's 24 MMAs in ~1150
        // clocks, little more than a thread needs to issue them.
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kM, kN, 0, 0);
            constexpr uint32_t idesc_o = idesc_f16_f32(kM, C::kOCols, 0, 1);   // P and V in fp16
            const uint64_t kdesc = smem_desc_sw128(sK, 16, 1024);
            const uint64_t vdesc = smem_desc_sw128(sV, C::kChunkBytes, 1024);
            const uint64_t qdesc = smem_desc_sw128(sQ, 16, 1024);
            auto issue_s = [&](int t, uint64_t kd) {
                const uint32_t tS = tmem + C::s_col(t);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
                    if constexpr (C::kQTmem)
                        mma_ts(tS, tmem + C::q_col(t) + kk * 8, kd + off, idesc_s, kk > 0 ? 1u : 0u);
                    else
                        mma_ss(tS, qdesc + (uint64_t)((t * C::kTileBytes) >> 4) + off, kd + off, idesc_s,
                               kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_s(t));
            };
            // PV_t in two halves of 64 keys (part 0: keys 0-63, issued as soon
            // as the softmax has written P for them; part 1 once all of P_t is
            // in), so that fewer MMAs stand between a finished softmax pass and
            // the next S_t.  Tiles on the causal diagonal carry the rows with
            // few visible keys, whose P entries are large: there P = P_hi +
            // P_lo (both fp16, P_lo in the upper 64 columns of the S region)
            // and a second MMA adds P_lo V.  A tile that is partial only
            // because its shard ends inside it needs the key mask alone: its
            // rows see every key of the other tiles as well.
            // (part 0: keys 0-63, part 1: keys 64-127, part -1: all keys)
            // `fresh`: O_t starts from zero with this tile (the first tile
            // overall; in the partials mode the first tile of every KV shard)
            auto issue_pv = [&](int t, uint64_t vd, bool fresh, bool split, int part) {
                const uint32_t tS = tmem + C::s_col(t), tO = tmem + C::o_col(t);
                const int k0 = part == 1 ? kN / 32 : 0, k1 = part == 0 ? kN / 32 : kN / 16;
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk)
                    if (kk >= k0 && kk < k1)
                        mma_ts(tO, tS + kk * 8, vd + (uint64_t)(kk * 128), idesc_o, (!fresh || kk > 0) ? 1u : 0u);
                if (split) {
#pragma unroll
                    for (int kk = 0; kk < kN / 16; ++kk)
                        if (kk >= k0 && kk < k1)
                            mma_ts(tO, tS + kN / 2 + kk * 8, vd + (uint64_t)(kk * 128), idesc_o, 1u);
                }
            };
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            tc_fence_after();
            int j = 0;
            bool split_prev[kNQ] = {false, false};
            bool fresh_prev = true;
            // PV_t(j-1) once P_t(j-1) is written (in two halves at d = 64)
            auto pv_when_ready = [&](int t, uint64_t vd, int jj) {
                const bool fresh = kMode == kParts ? fresh_prev : jj == 0;
                if constexpr (C::kHalfP) {
                    ok = mbar_wait(bar_pa(t), jj & 1, abort_flag);
                    if (!ok) return;
                    tc_fence_after();
                    issue_pv(t, vd, fresh, split_prev[t], 0);
                }
                ok = mbar_wait(bar_p(t), jj & 1, abort_flag);
                if (!ok) return;
                tc_fence_after();
                issue_pv(t, vd, fresh, split_prev[t], C::kHalfP ? 1 : -1);
            };
            // One KV tile.  A tcgen05.commit costs the issuing thread about as
            // much as an MMA, so there are three per tile: S_0, S_1 (each also
            // covers the previous PV of its half, which the softmax relies on
            // before rescaling O) and the stage release.
            auto step = [&](bool split0, bool split1, bool fresh) {
                const int s = j % C::kStages;
                const uint64_t kd = kdesc + (uint64_t)(s * (C::kTileBytes >> 4));
                if constexpr (C::kStages > 2) {
                    ok = mbar_wait(bar_kv(s), (j / C::kStages) & 1, abort_flag);
                    if (!ok) return;
                    tc_fence_after();
                    if (j == 0) {
                        for (int t = 0; t < kNQ; ++t) issue_s(t, kd);
                    } else {
                        // V(j-1) landed with K(j-1), waited for one tile ago
                        const int sp = (j - 1) % C::kStages;
                        const uint64_t vd = vdesc + (uint64_t)(sp * (C::kVStageBytes >> 4));
                        for (int t = 0; t < kNQ && ok; ++t) {
                            pv_when_ready(t, vd, j - 1);
                            if (!ok) break;
                            issue_s(t, kd);
                        }
                        if (!ok) return;
                        mma_commit(bar_e(sp));
                    }
                } else {
                    // Two K/V stages (d = 128): PV_0(j-1) needs only P_0(j-1) and
                    // V(j-1), so it goes ahead of the wait for K(j), and the stage of
                    // tile j-1 is released right after PV_1(j-1), its last reader, so
                    // that the producer refills it while S_1(j) runs; otherwise the
                    // next tile's load (~1000 clocks) starts only after every MMA of
                    // this tile, and the tensor pipe idles while it lands.
                    auto wait_kv = [&] {
                        ok = mbar_wait(bar_kv(s), (j / C::kStages) & 1, abort_flag);
                        if (ok) tc_fence_after();
                    };
                    if (j == 0) {
                        wait_kv();
                        if (!ok) return;
                        for (int t = 0; t < kNQ; ++t) issue_s(t, kd);
                    } else {
                        const int sp = (j - 1) % C::kStages;
                        const uint64_t vd = vdesc + (uint64_t)(sp * (C::kVStageBytes >> 4));
                        for (int t = 0; t < kNQ && ok; ++t) {
                            pv_when_ready(t, vd, j - 1);
                            if (!ok) break;
                            if (t == 0) {
                                wait_kv();
                                if (!ok) break;
                            }
                            if (t == kNQ - 1) mma_commit(bar_e(sp));
                            issue_s(t, kd);
                        }
                        if (!ok) return;
                    }
                }
                split_prev[0] = split0;
                split_prev[1] = split1;
                fresh_prev = fresh;
                ++j;
            };
            if constexpr (!kSplit) {
                // every tile full and visible: the KV tiles are just counted
                const int nkv = p.kvtab.S / kN;
                for (int jj = 0; jj < nkv && ok; ++jj) step(false, false, jj == 0);
            } else {
                int prev_shard = -1;
                ring_walk<kN>(p.kvtab, qt.shard, [&](int js, int, int nk, int natk, bool) {
                    if (!ok || !active(nk, natk)) return;
                    step(half_kind(causal, nat_h[0], nq_h[0], natk, nk) == kPartial &&
                             on_diagonal(causal, nat_h[0], natk, nk),
                         half_kind(causal, nat_h[1], nq_h[1], natk, nk) == kPartial &&
                             on_diagonal(causal, nat_h[1], natk, nk),
                         js != prev_shard);
                    prev_shard = js;
                });
            }
            if (ok && j > 0) {
                const int sp = (j - 1) % C::kStages;
                const uint64_t vd = vdesc + (uint64_t)(sp * (C::kVStageBytes >> 4));
                for (int t = 0; t < kNQ && ok; ++t) {
                    pv_when_ready(t, vd, j - 1);
                    if (!ok) break;
                    mma_commit(bar_o(t));   // the epilogue's single wait on O_t
                }
                if (ok) mma_commit(bar_e(sp));
            }
            // Every MMA issued above must finish before the TMEM is released.
            mma_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax + epilogue
        const int t = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t tS = lane_base + C::s_col(t);
        const uint32_t tO = lane_base + C::o_col(t);
        const int nq = nq_h[t];
        const int natq = nat_h[t] + row;
        const float sl2 = p.scale_log2;
        if constexpr (C::kQTmem) {
            // this thread's Q row -> TMEM (rows past the tile end are zero)
            uint32_t qr[D / 2];
            const int64_t goff = (((int64_t)b * p.tab.S + qt.row0 + kM * t + row) * H + h) * D;
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + goff);
#pragma unroll
            for (int u = 0; u < D / 8; ++u) {
                const uint4 x = row < nq ? src[u] : make_uint4(0u, 0u, 0u, 0u);
                qr[4 * u] = x.x;
                qr[4 * u + 1] = x.y;
                qr[4 * u + 2] = x.z;
                qr[4 * u + 3] = x.w;
            }
            tmem_st32(lane_base + C::q_col(t), qr);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q);
        }
        // one arrival per warp: every lane's tensor-memory stores are complete
        // (tcgen05.wait::st + fence by each lane, then the warp converges)
        auto warp_arrive = [&](uint32_t bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        float m = -INFINITY, l = 0.f;
        int j = 0;
        bool ok = true;
        // O_t (and its row-sum column) times alpha when the running max has
        // grown.  O_t already holds every previous PV product: PV_t(j-1) was
        // issued before S_t(j), and the commit that signalled S_t(j) covers all
        // earlier MMAs of the issuing thread.
        auto rescale_o = [&](float alpha) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                tmem_st32(tO + c * 32, r);
            }
            if constexpr (C::kSumCol) {
                uint32_t r[16];
                tmem_ld16(tO + D, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                tmem_st16(tO + D, r);
            }
        };
        // Partials mode: normalise and write this half's state as the partial of
        // KV shard js (have = false: the shard had no tile for this CTA, so the
        // partial is empty: O = 0, lse = -inf).  With have, O_t must hold every
        // PV product of the shard (the caller has waited for them).
        auto emit_part = [&](int js, bool have) {
            float lsum = 0.f;
            if (have) {
                if constexpr (C::kSumCol) {
                    uint32_t r[16];
                    tmem_ld16(tO + D, r);
                    tmem_wait_ld();
                    lsum = __uint_as_float(r[0]);
                } else {
                    lsum = l;
                }
            }
            const float inv = lsum > 0.f ? ldexpf(1.f, p.exps[0]) / lsum : 0.f;
            const int64_t grow = qt.row0 + kM * t + row;
            float* dst = p.part_out + ((((int64_t)js * p.B + b) * p.tab.S + grow) * H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                if (have) {
                    tmem_ld32(tO + c * 32, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = 0u;
                }
                if (row < nq) {
                    float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                            __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
                }
            }
            if (row < nq)
                p.part_lse[(((int64_t)js * p.B + b) * H + h) * p.tab.S + grow] =
                    lsum > 0.f ? (m + log2f(lsum)) * kLn2 : -INFINITY;
        };
        int cur_shard = -1;   // partials mode: the KV shard whose state O_t, m, l hold
        auto step = [&](int js, int nk, int natk) {
            if (!ok || !active(nk, natk)) return;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_s(t), j & 1, abort_flag));
            if (!ok) return;
            tc_fence_after();
            if constexpr (kMode == kParts) {
                if (js != cur_shard) {
                    // first tile of a new KV shard: S_t's completion also covers
                    // every PV of the previous shard, so O_t holds its whole sum
                    if (cur_shard >= 0) emit_part(cur_shard, true);
                    m = -INFINITY;
                    l = 0.f;
                    cur_shard = js;
                }
            }
            const int kind = half_kind(causal, nat_h[t], nq, natk, nk);
            bool resc = false;
            float alpha = 1.f;
            if (kind == kSkip) {
                uint32_t z[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_st16(tS + c * 16, z);
                if constexpr (C::kHalfP) {
                    tmem_wait_st();
                    tc_fence_before();
                    warp_arrive(bar_pa(t));
                }
            } else {
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
                tmem_wait_ld();
                int limit = nk - 1;   // the last key this row sees in the tile
                if (causal) limit = min(limit, natq - natk);
                if (kind == kPartial) {
#pragma unroll
                    for (int c = 0; c < kN; ++c)
                        if (c > limit) sr[c >> 5][c & 31] = 0xff800000u;   // -inf
                }
                // row max: four independent max3 chains of 16 steps each
                float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < kN; c += 8) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        mxa[u] = max3(mxa[u], __uint_as_float(sr[c >> 5][(c + 2 * u) & 31]),
                                      __uint_as_float(sr[c >> 5][(c + 2 * u + 1) & 31]));
                }
                const float mx = max3(mxa[0], mxa[1], fmaxf(mxa[2], mxa[3])) * sl2;
                float m_use = m;
                if (m == -INFINITY) {
                    m_use = mx;
                } else if (mx - m > kRescaleLog2) {
                    m_use = mx;
                    resc = true;
                    alpha = ex2(m - mx);
                }
                const float m_ref = m_use == -INFINITY ? 0.f : m_use;
                // p = 2^(s * scale * log2 e - m): one packed FMA per two scores,
                // one MUFU ex2 per score, one packed add per two scores.
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
                uint64_t acc0 = 0, acc1 = 0;   // two packed partial sums (0.0f bits)
                // The ordinary pass; tiles on the causal diagonal write P =
                // P_hi + P_lo, both fp16 (see issue_pv), in diag_pass.
                auto exp_pass = [&] {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (C::kHalfP && c == 2) {
                            // keys 0-63 are written: O_t is rescaled first (PV_t(j)
                            // must not have added to it yet), then PV_t may start on them
                            if (__any_sync(0xffffffffu, resc) && j > 0) rescale_o(alpha);
                            tmem_wait_st();
                            tc_fence_before();
                            warp_arrive(bar_pa(t));
                        }
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint64_t x = ffma2(
                                f2_pack(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sl2x2, negm2);
                            float x0, x1;
                            f2_unpack(x, x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            if constexpr (!C::kSumCol) {   // d = 64 sums in the MMA
                                if (i & 1)
                                    acc1 = fadd2(acc1, f2_pack(p0, p1));
                                else
                                    acc0 = fadd2(acc0, f2_pack(p0, p1));
                            }
                            pk[i] = pack_f16(p0, p1);
                        }
                        tmem_st16(tS + c * 16, pk);
                    }
                };
                bool diag = false;
                if constexpr (kSplit) diag = kind == kPartial && on_diagonal(causal, nat_h[t], natk, nk);
                if (diag) {
                    if constexpr (C::kHalfP) {
                        // O_t is rescaled before PV_t(j) may start on keys 0-63
                        if (__any_sync(0xffffffffu, resc) && j > 0) rescale_o(alpha);
                    }
                    const float tile_sum = diag_pass<!C::kSumCol, C::kHalfP>(tS, sl2, m_ref, limit, bar_pa(t));
                    if constexpr (!C::kSumCol) l = l * alpha + tile_sum;
                } else {
                    exp_pass();
                    float a0, a1, b0, b1;
                    if constexpr (!C::kSumCol) {
                        f2_unpack(acc0, a0, a1);
                        f2_unpack(acc1, b0, b1);
                        l = l * alpha + ((a0 + a1) + (b0 + b1));
                    }
                }
                m = m_use;
            }
            if constexpr (!C::kHalfP) {
                if (__any_sync(0xffffffffu, resc) && j > 0) rescale_o(alpha);
            }
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(bar_p(t));
            ++j;
        };
        if constexpr (!kSplit) {
            // every tile full and visible (the issuer counts them the same way)
            const int nkv = p.kvtab.S / kN;
            for (int jj = 0; jj < nkv && ok; ++jj) step(0, kN, 0);
        } else {
            ring_walk<kN>(p.kvtab, qt.shard, [&](int js, int, int nk, int natk, bool last) {
                step(js, nk, natk);
                if constexpr (kMode == kParts) {
                    if (ok && last && cur_shard != js) emit_part(js, false);
                }
            });
        }
        if (ok && j > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_o(t), 0, abort_flag));
        if constexpr (kMode == kParts) {
            if (ok && cur_shard >= 0) {
                tc_fence_after();
                emit_part(cur_shard, true);
            }
        } else if (ok) {
            tc_fence_after();
            if constexpr (C::kSumCol) {   // l = sum_j P_ij from O's extra column
                uint32_t r[16];
                tmem_ld16(tO + D, r);
                tmem_wait_ld();
                l = j > 0 ? __uint_as_float(r[0]) : 0.f;
            }
            // O holds P (V * 2^-e_v): undo the fp16 scaling of V with the normalisation
            float inv = l > 0.f ? ldexpf(1.f, p.exps[0]) / l : 0.f;
            const int64_t grow = qt.row0 + kM * t + row;
            const int64_t off = (((int64_t)b * p.tab.S + grow) * H + h) * D;
            const int64_t lse_at = ((int64_t)b * H + h) * p.tab.S + grow;
            float lse_out = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            // Ring step: merge with the running state (O_p, lse_p) by the log-sum-exp
            // rule, L = log(e^lse_p + e^lse), O = e^(lse_p - L) O_p + e^(lse - L) O.
            float w_prev = 0.f;
            if (kMode == kMerge && row < nq) {
                const float lp = p.prev_lse[lse_at];
                const float mx = fmaxf(lp, lse_out);
                if (mx == -INFINITY) {
                    inv = 0.f;
                } else {
                    const float a = exp2f((lp - mx) * kLog2e), c = exp2f((lse_out - mx) * kLog2e);
                    const float tot = a + c;
                    w_prev = a / tot;
                    inv *= c / tot;
                    lse_out = mx + logf(tot);
                }
            }
            const float* prow = p.prev_out + (kMode == kMerge ? off : 0);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + c * 32, r);
                tmem_wait_ld();
                if (kMode == kMerge && w_prev > 0.f) {
                    const float4* p4 = reinterpret_cast<const float4*>(prow + c * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 x = p4[i];
                        r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) * inv + w_prev * x.x);
                        r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) * inv + w_prev * x.y);
                        r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) * inv + w_prev * x.z);
                        r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) * inv + w_prev * x.w);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * inv);
                }
                if (row < nq) {
                    if (p.out_f32) {
                        float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                    } else {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                        uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + off + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
            if (row < nq) p.lse[lse_at] = lse_out;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
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

// BSHD bf16 tensor as a 4-D map (d, H, S, B), box (64, 1, 128, 1), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int B, int S, int H, int d,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)S * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool kSplit, int kMode, bool kHeads = false>
int launch_t(const st_layout& L, const st_layout& Lkv, const AttnArgs& a, void* stream, int t0, int t1) {
    using C = Cfg<D>;
    std::conditional_t<kHeads, FwdParamsHeads, FwdParams> p;
    const int S = (int)L.S, Skv = (int)Lkv.S;
    if (!make_map(&p.tq, a.q, a.B, S, a.H, D) || !make_map(&p.tk, a.k, a.B, Skv, a.H, D) ||
        !make_map(&p.tv, a.v16, a.B, Skv, a.H, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
        return (int)cudaErrorInvalidValue;
    fill_segtable(L, kNQ * kM, &p.tab);
    fill_segtable(Lkv, kN, &p.kvtab);
    if (t1 < 0 || t1 > p.tab.ntiles) t1 = p.tab.ntiles;
    if (t0 < 0) t0 = 0;
    if (t0 >= t1) return 0;
    p.tile0 = t0;
    // Longest-processing-time-first order for causal work: a 256-row unit
    // ending at natural position e sees about e keys.  Units of one head are
    // issued heaviest first; heads stay in order (grid y) for L2 reuse of K/V.
    p.use_order = 0;
    if (a.causal && t1 - t0 <= kMaxOrder) {
        std::vector<std::pair<int, int>> w;
        w.reserve(p.tab.ntiles);
        for (int s = 0; s < p.tab.nseg; ++s) {
            const int len = p.tab.seg_buf[s + 1] - p.tab.seg_buf[s];
            for (int tl = p.tab.seg_tile[s]; tl < p.tab.seg_tile[s + 1]; ++tl) {
                if (tl < t0 || tl >= t1) continue;
                const int local = (tl - p.tab.seg_tile[s]) * kNQ * kM;
                const int nq = std::min(kNQ * kM, len - local);
                w.emplace_back(-(p.tab.seg_nat[s] + local + nq), tl);
            }
        }
        std::stable_sort(w.begin(), w.end(),
                         [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first < y.first; });
        for (int i = 0; i < t1 - t0; ++i) p.order[i] = (uint16_t)w[i].second;
        p.use_order = 1;
    }
    p.q = a.q;
    p.out = a.out;
    p.out_f32 = a.out_dtype == ST_DTYPE_F32 ? 1 : 0;
    p.exps = a.exps;
    p.lse = a.lse;
    p.part_out = a.part_out;
    p.part_lse = a.part_lse;
    p.prev_out = a.prev_out;
    p.prev_lse = a.prev_lse;
    p.B = a.B;
    p.H = a.H;
    int hn = a.H;
    if constexpr (kHeads) {
        p.h0 = a.h0;
        p.hn = hn = a.hn;
    }
    p.scale_log2 = a.scale * kLog2e;
    p.causal = a.causal;
    auto kern = fwd_tc_kernel<D, kSplit, kMode, kHeads>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(t1 - t0, a.B * hn);
    kern<<<grid, kThreads, C::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int fwd_tc_tile_rows() { return kNQ * kM; }

int launch_fwd_tc2(const st_layout& L, const st_layout& Lkv, const AttnArgs& a, void* stream, int t0, int t1) {
    // partial (query half, KV tile) pairs exist under causal masking or when a
    // KV segment is not a multiple of the 128-key tile
    bool split = a.causal != 0;
    for (size_t s = 0; s + 1 < Lkv.seg_buf.size(); ++s)
        split |= ((Lkv.seg_buf[s + 1] - Lkv.seg_buf[s]) % kN) != 0;
    // a head range (h0, hn): the fused forward of the host-buffer entry point only
    const bool heads = a.hn > 0 && a.hn < a.H;
    if (heads && (a.part_out || a.prev_out || a.h0 < 0 || a.h0 + a.hn > a.H)) return (int)cudaErrorInvalidValue;
    if (heads) {
        if (a.d == 64)
            return split ? launch_t<64, true, kFused, true>(L, Lkv, a, stream, t0, t1)
                         : launch_t<64, false, kFused, true>(L, Lkv, a, stream, t0, t1);
        return split ? launch_t<128, true, kFused, true>(L, Lkv, a, stream, t0, t1)
                     : launch_t<128, false, kFused, true>(L, Lkv, a, stream, t0, t1);
    }
    if (a.part_out) {
        // partials: the ring walk of the split kernel, state written per KV shard
        return a.d == 64 ? launch_t<64, true, kParts>(L, Lkv, a, stream, t0, t1)
                         : launch_t<128, true, kParts>(L, Lkv, a, stream, t0, t1);
    }
    if (a.prev_out) {
        // ring step merged into the running state
        return a.d == 64 ? launch_t<64, true, kMerge>(L, Lkv, a, stream, t0, t1)
                         : launch_t<128, true, kMerge>(L, Lkv, a, stream, t0, t1);
    }
    if (a.d == 64)
        return split ? launch_t<64, true, kFused>(L, Lkv, a, stream, t0, t1)
                     : launch_t<64, false, kFused>(L, Lkv, a, stream, t0, t1);
    return split ? launch_t<128, true, kFused>(L, Lkv, a, stream, t0, t1)
                 : launch_t<128, false, kFused>(L, Lkv, a, stream, t0, t1);
}

int launch_fwd_tc(const st_layout& L, const AttnArgs& a, void* stream, bool* handled, int t0, int t1) {
    *handled = true;
    return launch_fwd_tc2(L, L, a, stream, t0, t1);
}

int fwd_tc_device_error(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(tc::g_device_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace st
