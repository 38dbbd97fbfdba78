// Backward sharded ring attention on tcgen05 tensor cores (sm_103a): bf16 in,
// fp16 tensor-core operands (exact scaled copies, see BwdParams), fp32
// accumulation, dK / dV in the gradient dtype, dQ accumulated in fp32.
//
// KV-stationary: one CTA owns a 128-key tile of one (batch, head) -- its K and
// V stay in shared memory and its dK, dV accumulate in tensor memory -- and
// walks the 128-row query tiles that see it in ring order: the query shards
// j, j+1, ..., j-1 (mod D) met by KV shard j as it travels around a ring
// (ShardTensor summary, section 4, ring attention, training).  For each query
// tile, with P = exp(scale S - lse) recomputed from the saved lse:
//
//   S^T  = K Q^T            (tcgen05.mma, smem x smem -> TMEM)
//   dP^T = V dO^T           (tcgen05.mma, smem x smem -> TMEM)
//   P^T, dS^T = P^T o (dP^T - Delta)   (softmax warps; P^T fp16 -> TMEM,
//                                       dS^T fp16 -> swizzled smem)
//   dV  += P^T dO           (A = P^T from TMEM)
//   dK  += dS^T Q           (A = dS^T, K-major view of the smem tile)
//   dQ_t = dS K             (A = dS, MN-major view of the same smem tile)
//   dQ  += scale dQ_t       (softmax warps: TMEM -> the dS^T lo tile -> TMA bulk reduction)
//
// Warp roles (384 threads): warp 0 TMA producer (+ lse / Delta staging),
// warp 1 TMEM allocator + MMA issuer (at d = 64 with warp 2 as a second
// issuer: dP^T and dK), warps 4-7 softmax for query columns 0-63 (one key row
// per thread), half of the dQ reduction (one query row per thread) and the dV
// epilogue, warps 8-11 the same for columns 64-127 and the dK epilogue.
// Tensor memory: S^T|P^T, dP^T|dQ_t, dV, dK at d = 128; at d = 64 dQ_t has two
// buffers of its own after dK, and a tile's dQ drain runs after the next
// tile's softmax pass.  Every barrier wait is bounded (tc_ptx.cuh).
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <type_traits>
#include <vector>

#include "device.cuh"
#include "tc_ptx.cuh"

namespace st {
namespace {

using namespace tc;

constexpr int kT = 128;          // keys per CTA, rows per query tile
constexpr int kMaxOrder = 4096;  // longest tile order passed as a kernel parameter
constexpr int kFlush = 8;        // query tiles per TMEM accumulation segment (lead tile)
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kChunkBytes = kT * 128;             // 128 rows x 64 fp16
    static constexpr int kTileBytes = kChunks * kChunkBytes; // 128 rows x D fp16
    static constexpr int kStages = D == 64 ? 2 : 1;
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kTileBytes;
    static constexpr int kQOff = kVOff + kTileBytes;               // [stage] Q tiles
    static constexpr int kOOff = kQOff + kStages * kTileBytes;     // [stage] dO tiles
    static constexpr int kSOff = kOOff + kStages * kTileBytes;     // dS^T (hi), 128 x 128 fp16
    static constexpr int kS2Off = kSOff + 2 * kChunkBytes;         // dS^T lo part (split tiles)
    static constexpr int kLOff = kS2Off + 2 * kChunkBytes;         // [stage] lse*log2e, Delta
    // second dQ staging slice of each softmax warp (the first is its slice of the dS^T lo tile)
    static constexpr int kDq2Off = kLOff + kStages * 2 * kT * 4;
    static constexpr int kBarOff = kDq2Off + 8 * 4096;
    // kv_full, q_full[S], q_empty[S], s_full, ds_ready, it_done, dq_free, drain
    static constexpr int kNumBars = 6 + 2 * kStages;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;
    static constexpr uint32_t kColDP = 128;
    static constexpr uint32_t kColDV = 256;
    static constexpr uint32_t kColDK = 256 + D;
    // d = 64: dQ_t in two buffers of its own (columns 384-447, 448-511, by
    // query-tile parity), so the next dP^T need not wait for the drain, and the
    // drain of tile i can run after the softmax pass of tile i + 1.  At d = 128
    // dQ_t reuses the dP^T columns.
    static constexpr bool kOwnDq = D == 64;
    static constexpr uint32_t kColDQ = 256 + 2 * D;
    // d = 64: the MMAs are issued by two threads (warps 1 and 2), since one
    // thread issues an N = 64 MMA more slowly than the tensor core runs it;
    // the barriers the MMAs signal then count one commit from each.
    static constexpr bool kTwoIss = D == 64;
    static constexpr int kIss = kTwoIss ? 2 : 1;
};

// Operands: exact fp16 copies of q, k, v, dO scaled by 2^-e (e per tensor,
// chosen from its max |x|), so P and dS can be fed to the tensor cores in fp16
// (11 significant bits) rather than bf16 (8): P enters as P * 2^14 and dS as
// dS * 2^-e_dS, which keeps both inside fp16's normal range.  The scales are
// undone in fp32 when S, dP and the gradients leave tensor memory.
constexpr int kPShift = 14;

struct BwdParams {
    CUtensorMap tq;
    CUtensorMap tk;
    CUtensorMap tv;
    CUtensorMap tdo;
    CUtensorMap tdq;          // dq_acc, fp32, box 32 x 32 rows, 128-byte swizzle
    SegTable tab;             // 128-row key tiles (k, v, dk, dv)
    SegTable qtab;            // 128-row query tiles (q, dO, lse, Delta, dq): the same
                              // layout, or in a ring step another shard
    const float* lse;         // [B,H,S]
    const float* delta;       // [B,H,S]
    float* dq_acc;            // [B,S,H,D] fp32
    void* dk;
    void* dv;
    const int* exps;          // scale exponents of q, k, v, dO, dS
    int B, H;
    float scale;
    float scale_log2;
    int causal;
    int grad_f32;             // dK / dV written as fp32 (else bf16)
    int accum;                // ring step: dK / dV added into the fp32 outputs
    int use_order;            // causal: CTAs take key tiles heaviest first
    uint16_t order[kMaxOrder];
};

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

__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
    float4 x;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w) : "r"(addr)
                 : "memory");
    return x;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Walk the 128-row query tiles met by KV shard `j` in ring order: query shards
// j, j+1, ..., j-1 (mod D); f(row0, nq, nat0).
template <typename F>
__device__ __forceinline__ void ring_walk_q(const SegTable& T, int j, F&& f) {
    for (int t = 0; t < T.D; ++t) {
        int r = j + t;
        if (r >= T.D) r -= T.D;
        for (int s = T.shard_seg[r]; s < T.shard_seg[r + 1]; ++s) {
            const int b0 = T.seg_buf[s], b1 = T.seg_buf[s + 1], nat = T.seg_nat[s];
            for (int q0 = b0; q0 < b1; q0 += kT) f(q0, min(kT, b1 - q0), nat + (q0 - b0));
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ BwdParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (sbase - raw);
    const uint32_t sK = sbase + C::kKOff, sV = sbase + C::kVOff, sQ = sbase + C::kQOff,
                   sO = sbase + C::kOOff, sS = sbase + C::kSOff, sS2 = sbase + C::kS2Off;
    float* lse_s = reinterpret_cast<float*>(gbase + C::kLOff);   // [stage][2][128]
    const uint32_t bars = sbase + C::kBarOff;
    const uint32_t bar_kv = bars;
    auto bar_qf = [&](int s) { return bars + 8u * (1 + s); };
    auto bar_qe = [&](int s) { return bars + 8u * (1 + C::kStages + s); };
    const uint32_t bar_s = bars + 8u * (1 + 2 * C::kStages);
    const uint32_t bar_ds = bar_s + 8;
    const uint32_t bar_it = bar_s + 16;
    const uint32_t bar_dqf = bar_s + 24;
    const uint32_t bar_drain = bar_s + 32;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.H, S = p.tab.S, Sq = p.qtab.S;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int tile = p.use_order ? (int)p.order[blockIdx.x] : (int)blockIdx.x;
    const QTile kt = locate_qtile(p.tab, tile, kT);           // this CTA's key tile
    // Extra precision (hi + lo fp16 parts of P and dS) where gradients are
    // large compared with their RMS: tiles on the causal diagonal, which
    // hold the rows and keys with few partners, and under causal masking the
    // key tile holding the first natural positions, which every query attends
    // to (its dV and dK are orders of magnitude above the typical key's).
    const bool lead_tile = p.causal && kt.nat0 < kT;
    auto wants_split = [&](int kind, int natq) {
        return (kind == kPartial && on_diagonal(p.causal, natq, kt.nat0, kt.nq)) || lead_tile;
    };
    // fp32 gradients of the lead key tile: its dV and dK sum tens of thousands
    // of products, and the tensor core's fp32 accumulation of that many terms
    // drifts by ~1e-4 relative -- on the largest gradients of the tensor.  So
    // every kFlush query tiles the TMEM accumulators are added into the fp32
    // output rows (owned by this CTA) and the MMAs restart from zero.
    const bool flush_tile = lead_tile && p.grad_f32;
    auto seg_start = [&](int it) { return flush_tile ? (it % kFlush) == 0 : it == 0; };
    const int causal = p.causal;
    auto active = [&](int nq, int natq) {
        return classify(causal, natq, nq, kt.nat0, kt.nq, kT) != kSkip;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar_qf(s), 2);     // the TMA bytes' arrival + the producer warp's statistics
            mbar_init(bar_qe(s), C::kIss);
        }
        mbar_init(bar_s, C::kIss);
        mbar_init(bar_ds, 8);       // one arrival per softmax warp
        mbar_init(bar_it, C::kIss);
        mbar_init(bar_dqf, 8);
        mbar_init(bar_drain, C::kIss);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int64_t lse_base = ((int64_t)b * H + h) * Sq;

    if (warp == 0) {
        // ------------------------------------------------ producer
        uint32_t issued_tx = 0;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_4d(sK + c * C::kChunkBytes, &p.tk, bar_kv, c * 64, h, kt.row0, b);
                tma_load_4d(sV + c * C::kChunkBytes, &p.tv, bar_kv, c * 64, h, kt.row0, b);
            }
        }
        // Row statistics staged per query tile, in the form the softmax uses:
        //   [0, kT):   kPShift - lse * log2(e)   (-inf for rows past the tile)
        //   [kT, 2kT): -Delta * 2^-(e_dS + kPShift)
        const float ds_mul = ldexpf(1.f, -p.exps[4] - kPShift);
        int i = 0;
        bool ok = true;
        ring_walk_q(p.qtab, kt.shard, [&](int q0, int nq, int natq) {
            if (!ok || !active(nq, natq)) return;
            const int s = i % C::kStages;
            // fetched before the stage is free, so the global loads overlap the wait
            float nl[kT / 32], nd[kT / 32];
#pragma unroll
            for (int e = 0; e < kT / 32; ++e) {
                const int r = e * 32 + lane;
                const bool valid = r < nq;
                nl[e] = valid ? (float)kPShift - p.lse[lse_base + q0 + r] * kLog2e : -INFINITY;
                nd[e] = valid ? -p.delta[lse_base + q0 + r] * ds_mul : 0.f;
            }
            if (i >= C::kStages)
                ok = __all_sync(0xffffffffu, mbar_wait(bar_qe(s), ((i / C::kStages) - 1) & 1, abort_flag));
            if (!ok) return;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar_qf(s), 2 * C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_4d(sQ + s * C::kTileBytes + c * C::kChunkBytes, &p.tq, bar_qf(s), c * 64, h, q0, b);
                    tma_load_4d(sO + s * C::kTileBytes + c * C::kChunkBytes, &p.tdo, bar_qf(s), c * 64, h, q0, b);
                }
                issued_tx++;
            }
            float* ls = lse_s + s * 2 * kT;
#pragma unroll
            for (int e = 0; e < kT / 32; ++e) {
                ls[e * 32 + lane] = nl[e];
                ls[kT + e * 32 + lane] = nd[e];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qf(s));
            ++i;
        });
        if (lane == 0) {
            // every load issued lands before the CTA can exit (also after an abort)
            mbar_wait_drain(bar_kv, 0);
            for (int ii = max(0, i - C::kStages); ii < i; ++ii)
                mbar_wait_drain(bar_qf(ii % C::kStages), (ii / C::kStages) & 1);
        }
        (void)issued_tx;
    } else if (warp == 1 || (C::kTwoIss && warp == 2)) {
        // ------------------------------------------------ MMA issuer(s)
        // Two issuing threads at d = 64: warp 1 (role a) issues S^T, dV and
        // dQ_t, warp 2 dP^T and dK.  On tiles with hi + lo parts warp 1 also
        // issues dK, and the next dP^T (which overwrites the P_lo columns that
        // its dV MMAs read): the MMAs of one thread run in issue order, those of
        // two threads do not.  Every other shared operand or accumulator is
        // ordered through the barriers: a commit tracks all earlier MMAs of its
        // own thread, and each barrier waits for both threads' commits.
        const bool role_a = warp == 1;
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_f16_f32(kT, kT, 0, 0);      // S^T, dP^T
            constexpr uint32_t id_kv = idesc_f16_f32(kT, D, 0, 1);      // dV, dK (B MN-major)
            constexpr uint32_t id_q = idesc_f16_f32(kT, D, 1, 1);       // dQ (A and B MN-major)
            // Descriptors of every operand tile at offset 0, K-major (_k) and
            // MN-major (_mn) views; a stage or K step adds its byte offset >> 4
            // to the start-address field (the issuing thread's per-MMA work
            // is what bounds how fast the MMAs can be fed).
            const uint64_t k_k = smem_desc_sw128(sK, 16, 1024), k_mn = smem_desc_sw128(sK, C::kChunkBytes, 1024);
            const uint64_t v_k = smem_desc_sw128(sV, 16, 1024);
            const uint64_t q_k = smem_desc_sw128(sQ, 16, 1024), q_mn = smem_desc_sw128(sQ, C::kChunkBytes, 1024);
            const uint64_t o_k = smem_desc_sw128(sO, 16, 1024), o_mn = smem_desc_sw128(sO, C::kChunkBytes, 1024);
            const uint64_t ds_k[2] = {smem_desc_sw128(sS, 16, 1024), smem_desc_sw128(sS2, 16, 1024)};
            const uint64_t ds_mn[2] = {smem_desc_sw128(sS, C::kChunkBytes, 1024),
                                       smem_desc_sw128(sS2, C::kChunkBytes, 1024)};
            // K step kk of a K-major tile (two 64-column chunks) / of an MN-major tile (16 rows)
            auto koff = [](int kk) { return (uint64_t)(((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4); };
            auto moff = [](int kk) { return (uint64_t)(kk * (2048 >> 4)); };
            // TMEM column of P^T (P_lo) for K step kk: query columns 0-63 are
            // packed into columns 0-31, 64-127 into 64-95 (one softmax group each)
            auto pk = [](int kk) { return (uint32_t)(kk * 8 + (kk >> 2) * 32); };
            bool ok = mbar_wait(bar_kv, 0, abort_flag);
            tc_fence_after();
            int i = 0;
            bool prev_split = false;
            ring_walk_q(p.qtab, kt.shard, [&](int, int nq, int natq) {
                if (!ok || !active(nq, natq)) return;
                const int s = i % C::kStages;
                const uint64_t st = (uint64_t)(s * (C::kTileBytes >> 4));
                // S^T(i) overwrites P^T(i-1) and dP^T(i) overwrites P_lo(i-1),
                // both read by MMAs of iteration i-1 issued earlier (the
                // tcgen05.mma operations of one thread run in issue order); the
                // dP^T columns also hold dQ_t(i-1), so dP^T(i) waits for its drain.
                ok = mbar_wait(bar_qf(s), (i / C::kStages) & 1, abort_flag);
                if (!ok) return;
                tc_fence_after();
                if (role_a) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + C::kColS, k_k + koff(kk), q_k + st + koff(kk), id_s, kk > 0);
                }
                if (!C::kOwnDq && i > 0) {
                    ok = mbar_wait(bar_dqf, (i - 1) & 1, abort_flag);
                    if (!ok) return;
                    tc_fence_after();
                }
                if (!C::kTwoIss || role_a == prev_split) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem + C::kColDP, v_k + koff(kk), o_k + st + koff(kk), id_s, kk > 0);
                }
                mma_commit(bar_s);
                ok = mbar_wait(bar_ds, i & 1, abort_flag);
                if (!ok) return;
                tc_fence_after();
                // Tiles on the causal diagonal hold the pairs of rows and keys
                // with few partners, whose P and dS are large: there (and on
                // the lead key tile) both
                // are split into fp16 hi + lo parts (P_lo in the consumed dP^T
                // columns, dS_lo in a second smem tile) and every product gets
                // a second MMA for the lo part.
                const bool split = wants_split(classify(causal, natq, nq, kt.nat0, kt.nq, kT), natq);
                if (role_a) {
                    // dV += P^T dO  (A: P^T fp16 in TMEM; B: dO, K = query rows, N = D)
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)
                        mma_ts(tmem + C::kColDV, tmem + C::kColS + pk(kk), o_mn + st + moff(kk), id_kv,
                               (!seg_start(i) || kk > 0) ? 1u : 0u);
                    if (split) {
#pragma unroll
                        for (int kk = 0; kk < kT / 16; ++kk)
                            mma_ts(tmem + C::kColDV, tmem + C::kColDP + pk(kk), o_mn + st + moff(kk), id_kv, 1u);
                    }
                }
                // dK += dS^T Q  (A: dS^T K-major in smem; B: Q, K = query rows, N = D)
                if (!C::kTwoIss || role_a == split) {
                    for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
                        for (int kk = 0; kk < kT / 16; ++kk)
                            mma_ss(tmem + C::kColDK, ds_k[part] + koff(kk), q_mn + st + moff(kk), id_kv,
                                   (!seg_start(i) || kk > 0 || part > 0) ? 1u : 0u);
                    }
                }
                // Q(i) and dO(i) are read by no later MMA: the producer may refill
                // the stage while dQ_t runs.
                mma_commit(bar_qe(s));
                // dQ_t = dS K  (A: dS, M = query rows contiguous; B: K, K = keys, N = D).
                // d = 128: it overwrites the P_lo columns, which the dV MMA above
                // read first (tcgen05.mma operations of one thread run in order).
                // d = 64: buffer i & 1 of its own, whose previous tile (i - 2)
                // every softmax warp has drained before its "dS ready" arrival
                // of tile i (the drain of tile i - 2 precedes the pass of tile i).
                const uint32_t col_dq = C::kOwnDq ? C::kColDQ + (uint32_t)(i & 1) * D : C::kColDP;
                if (role_a) {
                    for (int part = 0; part < (split ? 2 : 1); ++part) {
#pragma unroll
                        for (int kk = 0; kk < kT / 16; ++kk)
                            mma_ss(tmem + col_dq, ds_mn[part] + moff(kk), k_mn + moff(kk), id_q,
                                   (kk > 0 || part > 0) ? 1u : 0u);
                    }
                }
                mma_commit(bar_it);
                prev_split = split;
                ++i;
            });
            mma_commit(bar_drain);
            mbar_wait_drain(bar_drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax, dQ reduction, epilogue
        // Two groups of four warps, one key row per thread in each: group 0
        // (warps 4-7) forms P^T and dS^T for query columns 0-63 and writes
        // dV; group 1 (warps 8-11) does query columns 64-127, writes dK, and
        // drains dQ_t (one query row per thread) after each tile's MMAs.
        const int grp = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int r = quad * 32 + lane;               // key row (softmax) / query row (dQ drain)
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        const int natk = kt.nat0 + r;
        const float sl2 = ldexpf(p.scale_log2, p.exps[0] + p.exps[1]);    // S' -> scaled log2 units
        const float sc = ldexpf(p.scale, p.exps[4] + p.exps[1]);           // dQ_t -> dQ
        // dQ staging: the 4 KB of the dS^T lo tile that this warp itself
        // writes -- its 32 key rows of its group's 64 columns.  The lo tile is
        // written only by the softmax passes of split tiles (the causal diagonal and
        // the lead key tile), so the next pass of an ordinary tile need not
        // wait for the TMA to have read the staged dQ out of it.
        const uint32_t stg = sS2 + (uint32_t)(grp * C::kChunkBytes + quad * 32 * 128);
        // the warp's second staging slice: successive dQ chunks alternate between
        // the two, so a chunk waits only for the TMA read of the chunk before the
        // previous one
        const uint32_t stg2 = sbase + C::kDq2Off + (uint32_t)((warp - 4) * 4096);
        int nch = 0;
        // Write (or, after a flush, add) this key row's dV (group 0) or
        // scale * dK (group 1) from the TMEM accumulator into the output.
        auto emit = [&](bool have, bool add) {
            const int64_t off = (((int64_t)b * S + kt.row0 + r) * H + h) * D;
            {
                const int which = grp;
                const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
                const float mul = which == 0 ? ldexpf(1.f, p.exps[3] - kPShift)
                                             : ldexpf(p.scale, p.exps[4] + p.exps[0]);
                void* dst = which == 0 ? p.dv : p.dk;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    if (have) {
                        tmem_ld32(lane_base + col + c * 32, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    if (r < kt.nq) {
                        if (p.grad_f32) {
                            float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(dst) + off + c * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                float4 x = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                                                       __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
                                if (add) {
                                    const float4 y = d4[e];
                                    x.x += y.x;
                                    x.y += y.y;
                                    x.z += y.z;
                                    x.w += y.w;
                                }
                                d4[e] = x;
                            }
                        } else {
                            uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + off + c * 32);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                d4[e] = make_uint4(
                                    pack_bf16(__uint_as_float(v[8 * e]) * mul, __uint_as_float(v[8 * e + 1]) * mul),
                                    pack_bf16(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul),
                                    pack_bf16(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul),
                                    pack_bf16(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul));
                        }
                    }
                }
            }
        };
        bool flushed = false;
        // dS' = P' (dP - Delta) 2^-(e_dS + kPShift), with the power of two
        // folded into dP's multiplier and into the staged -Delta
        const float dpm = ldexpf(1.f, p.exps[2] + p.exps[3] - p.exps[4] - kPShift);
        const uint64_t sl2x2 = f2_pack(sl2, sl2), dpm2 = f2_pack(dpm, dpm);
        // One query tile.  Compile-time variants: kMask (partial tiles: the
        // causal diagonal and ragged key tiles need a per-element mask; query
        // columns past the tile end are zeroed by their -inf statistic) and
        // kLo (hi + lo fp16 parts of P and dS, see the MMA issuer).
        // TMEM column of the packed P^T (or P_lo) for 32-column chunk c4
        auto pcol = [](int c4) { return (uint32_t)(c4 * 16 + (c4 >> 1) * 32); };
        auto tile_pass = [&](auto mask_tag, auto lo_tag, uint32_t ls, int cmin) {
            constexpr bool kMask = decltype(mask_tag)::value;
            constexpr bool kLo = decltype(lo_tag)::value;
            const bool row_ok = r < kt.nq;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c4 = 2 * grp + cc;   // this group's 32-column chunks
                uint32_t sv[32], dv[32];
                tmem_ld32(lane_base + C::kColS + c4 * 32, sv);
                tmem_ld32(lane_base + C::kColDP + c4 * 32, dv);
                tmem_wait_ld();
                uint32_t pp[16], dd[16], pl[16], dl[16];
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2) {
                    // statistics of columns c .. c+3 (broadcast shared loads)
                    const int c = c4 * 32 + 4 * e2;
                    const float4 nl = ld_shared_v4f(ls + (uint32_t)(c * 4));
                    const float4 nd = ld_shared_v4f(ls + (uint32_t)((kT + c) * 4));
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int e = 2 * e2 + h2;
                        const uint64_t nl2 = h2 ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y);
                        const uint64_t nd2 = h2 ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y);
                        float x0, x1;
                        f2_unpack(ffma2(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2x2, nl2),
                                  x0, x1);
                        float p0 = ex2(x0), p1 = ex2(x1);
                        if constexpr (kMask) {
                            // query column cc is visible to this key iff cc >= cmin (and the key row exists)
                            if (!row_ok || c + 2 * h2 < cmin) p0 = 0.f;
                            if (!row_ok || c + 2 * h2 + 1 < cmin) p1 = 0.f;
                        }
                        const uint64_t p2 = f2_pack(p0, p1);
                        const uint64_t t2 =
                            ffma2(f2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), dpm2, nd2);
                        float d0, d1;
                        f2_unpack(fmul2(p2, t2), d0, d1);
                        pp[e] = pack_f16(p0, p1);
                        dd[e] = pack_f16(d0, d1);
                        if constexpr (kLo) {
                            const float2 ph = __half22float2(*reinterpret_cast<const __half2*>(&pp[e]));
                            const float2 dh = __half22float2(*reinterpret_cast<const __half2*>(&dd[e]));
                            pl[e] = pack_f16(p0 - ph.x, p1 - ph.y);
                            dl[e] = pack_f16(d0 - dh.x, d1 - dh.y);
                        }
                    }
                }
                // P^T chunk -> S columns this group has already read (query
                // columns 0-63 -> columns 0-31, 64-127 -> 64-95); P_lo likewise
                // into the dP^T columns
                tmem_st16(lane_base + C::kColS + pcol(c4), pp);
                if constexpr (kLo) tmem_st16(lane_base + C::kColDP + pcol(c4), pl);
                // dS^T columns c4*32 .. +31 = 16-byte units 4*(c4&1) .. +3 of chunk c4>>1
                const uint32_t coff = (uint32_t)r * 128 + (uint32_t)(c4 >> 1) * C::kChunkBytes;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)((c4 & 1) * 4 + u);
                    const uint32_t at = coff + ((unit ^ (uint32_t)(r & 7)) << 4);
                    st_shared_v4(sS + at, dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
                    if constexpr (kLo)
                        st_shared_v4(sS2 + at, dl[4 * u], dl[4 * u + 1], dl[4 * u + 2], dl[4 * u + 3]);
                }
            }
        };
        // dQ_t of the tile whose MMAs just finished -> dq_acc (group 1)
        // dQ_t of the tile whose MMAs just finished -> dq_acc; each group
        // takes half of the columns (one query row per thread)
        // `it`: the tile's index among the active ones (its dQ_t buffer at d = 64);
        // `late`: the drain runs after the next tile's softmax pass (d = 64), while
        // that tile's MMAs may read the dS^T lo tile, so it stages only in the
        // warp's own slice.
        auto drain = [&](int q0, int nq, int it, bool late) {
            // This group's columns of the row come into registers first and
            // the TMEM is released at once (at d = 128 the next dP^T waits for
            // both groups); the reductions then overlap the MMAs.
            constexpr int kCols = D / 2;
            const uint32_t col = C::kOwnDq ? C::kColDQ + (uint32_t)(it & 1) * D : C::kColDP;
            uint32_t v[kCols];
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c)
                tmem_ld32(lane_base + col + grp * kCols + c * 32, *reinterpret_cast<uint32_t(*)[32]>(v + c * 32));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (!C::kOwnDq && lane == 0) mbar_arrive(bar_dqf);
            // The reductions go through the TMA: per 32-column chunk the warp
            // writes its 32 rows into a 128-byte-swizzled fp32 tile (rows past
            // the query tile as zeros, which add nothing) and one lane issues a
            // bulk tensor reduction (add) into dq_acc; the warp then goes on to
            // its next softmax pass while the reductions run.
            const bool row_ok = quad * 32 + lane < nq;
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c) {
                // the TMA has read this slice's previous chunk out of it; the other
                // slice's (most recent) group may still be reading.  A late drain
                // uses only the warp's own slice.
                if (lane == 0) {
                    if (late)
                        bulk_wait_read_0();
                    else
                        bulk_wait_read_1();
                }
                __syncwarp();
                const uint32_t buf = late ? stg2 : ((nch++ & 1) ? stg2 : stg);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    // 16-byte unit k of row `lane` under the 128-byte swizzle
                    const uint32_t unit = (uint32_t)(k ^ (lane & 7));
                    const int e = c * 32 + 4 * k;
                    st_shared_v4(buf + (uint32_t)(lane * 128) + unit * 16,
                                 row_ok ? __float_as_uint(__uint_as_float(v[e]) * sc) : 0u,
                                 row_ok ? __float_as_uint(__uint_as_float(v[e + 1]) * sc) : 0u,
                                 row_ok ? __float_as_uint(__uint_as_float(v[e + 2]) * sc) : 0u,
                                 row_ok ? __float_as_uint(__uint_as_float(v[e + 3]) * sc) : 0u);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_4d(&p.tdq, buf, grp * kCols + c * 32, h, q0 + quad * 32, b);
                    bulk_commit_group();
                }
            }
        };
        // d = 64 (unless the CTA flushes its accumulators): the drain of tile i
        // runs after the softmax pass of tile i + 1, while that tile's MMAs run.
        // Waiting for S^T and dP^T of tile i + 1 also waits for every MMA of
        // tile i (a commit tracks all earlier MMAs of its thread).
        const bool late = C::kOwnDq && !flush_tile;
        int pq0 = 0, pnq = 0;    // the tile whose drain is pending (late)
        int i = 0;
        bool ok = true;
        ring_walk_q(p.qtab, kt.shard, [&](int q0, int nq, int natq) {
            if (!ok || !active(nq, natq)) return;
            if (flush_tile && i > 0 && (i % kFlush) == 0) {
                // promote the finished segment (all MMAs of iteration i-1 done:
                // waited for in the drain)
                tc_fence_after();
                emit(true, flushed || p.accum);
                flushed = true;
            }
            const int s = i % C::kStages;
            ok = __all_sync(0xffffffffu, mbar_wait(bar_qf(s), (i / C::kStages) & 1, abort_flag));
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_s, i & 1, abort_flag));
            if (!ok) return;
            tc_fence_after();
            // this stage's row statistics (shared-memory address)
            const uint32_t ls = sbase + C::kLOff + (uint32_t)(s * 2 * kT * 4);
            const int kind = classify(causal, natq, nq, kt.nat0, kt.nq, kT);
            // a pass that writes the lo tile waits until the TMA has read the
            // dQ staged in this warp's slice of it
            const bool lo = wants_split(kind, natq);
            if (lo) {
                if (lane == 0) bulk_wait_read_0();
                __syncwarp();
            }
            if (kind == kPartial) {
                // causal: query column c sees key natk iff natk <= natq + c
                const int cmin = causal ? max(0, natk - natq) : 0;
                if (lo)
                    tile_pass(std::true_type{}, std::true_type{}, ls, cmin);
                else
                    tile_pass(std::true_type{}, std::false_type{}, ls, cmin);
            } else if (lead_tile) {
                tile_pass(std::false_type{}, std::true_type{}, ls, 0);
            } else {
                tile_pass(std::false_type{}, std::false_type{}, ls, 0);
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_ds);
            if (late) {
                if (i > 0) drain(pq0, pnq, i - 1, true);
                pq0 = q0;
                pnq = nq;
            } else {
                ok = __all_sync(0xffffffffu, mbar_wait(bar_it, i & 1, abort_flag));
                if (!ok) return;
                tc_fence_after();
                drain(q0, nq, i, false);
            }
            ++i;
        });
        if (ok && late && i > 0) {
            // the last tile: all MMAs of the CTA done (the issuer's final
            // commit, a barrier of a single phase)
            ok = __all_sync(0xffffffffu, mbar_wait(bar_drain, 0, abort_flag));
            if (ok) {
                tc_fence_after();
                drain(pq0, pnq, i - 1, true);
            }
        }
        // epilogue: dV (group 0) or scale * dK (group 1) for this key row (the
        // last tile's MMAs were waited for before its drain)
        if (ok) {
            tc_fence_after();
            emit(i > 0, flushed || p.accum);
        }
        // the staged dQ reductions have completed before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
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

// BSHD fp16 tensor as a 4-D map (d, H, S, B), box (64, 1, 128, 1), 128-byte swizzle.
// dq_acc (fp32 [B,S,H,d]) as a 4-D map (d, H, S, B), box (32, 1, 32, 1), 128-byte
// swizzle: the tile one dQ-reducing warp adds per chunk.
bool make_map_dq(CUtensorMap* m, void* base, int B, int S, int H, int d) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 4, (cuuint64_t)H * d * 4, (cuuint64_t)S * H * d * 4};
    const cuuint32_t box[4] = {32, 1, 32, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map(CUtensorMap* m, const void* base, int B, int S, int H, int d) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)S * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_t(const st_layout& Lq, const st_layout& L, const BwdArgs& a, void* stream) {
    using C = Cfg<D>;
    BwdParams p;
    const int Sq = (int)Lq.S, S = (int)L.S;
    if (!make_map(&p.tq, a.h16[0], a.B, Sq, a.H, D) || !make_map(&p.tk, a.h16[1], a.B, S, a.H, D) ||
        !make_map(&p.tv, a.h16[2], a.B, S, a.H, D) || !make_map(&p.tdo, a.h16[3], a.B, Sq, a.H, D) ||
        !make_map_dq(&p.tdq, a.dq_acc, a.B, Sq, a.H, D))
        return (int)cudaErrorInvalidValue;
    fill_segtable(L, kT, &p.tab);
    fill_segtable(Lq, kT, &p.qtab);
    // Longest-processing-time-first order for causal work: a key tile starting
    // at natural position n is seen by about S - n query rows.
    p.use_order = 0;
    if (a.causal && p.tab.ntiles <= kMaxOrder) {
        std::vector<std::pair<int, int>> w;
        w.reserve(p.tab.ntiles);
        for (int s = 0; s < p.tab.nseg; ++s)
            for (int tl = p.tab.seg_tile[s]; tl < p.tab.seg_tile[s + 1]; ++tl)
                w.emplace_back(p.tab.seg_nat[s] + (tl - p.tab.seg_tile[s]) * kT, tl);
        std::stable_sort(w.begin(), w.end(),
                         [](const std::pair<int, int>& x, const std::pair<int, int>& y) { return x.first < y.first; });
        for (int i = 0; i < p.tab.ntiles; ++i) p.order[i] = (uint16_t)w[i].second;
        p.use_order = 1;
    }
    p.lse = a.lse;
    p.delta = a.delta;
    p.dq_acc = a.dq_acc;
    p.dk = a.dk;
    p.dv = a.dv;
    p.exps = a.exps;
    p.B = a.B;
    p.H = a.H;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.causal = a.causal;
    p.grad_f32 = a.grad_dtype == ST_DTYPE_F32 ? 1 : 0;
    p.accum = a.accum && p.grad_f32 ? 1 : 0;
    auto kern = bwd_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(p.tab.ntiles, a.B * a.H);
    kern<<<grid, kThreads, C::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(p);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_bwd_tc2(const st_layout& Lq, const st_layout& Lkv, const BwdArgs& a, void* stream) {
    return a.d == 64 ? launch_t<64>(Lq, Lkv, a, stream) : launch_t<128>(Lq, Lkv, a, stream);
}

int launch_bwd_tc(const st_layout& L, const BwdArgs& a, void* stream, bool* handled) {
    *handled = true;
    return launch_bwd_tc2(L, L, a, stream);
}

int bwd_tc_device_error(bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, tc::g_device_error, sizeof(int)) != cudaSuccess) return -1;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(tc::g_device_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace st
