// Internal declarations shared by the host layout code, the C-ABI layer and
// the kernels.  Not part of the public interface (include/st_attn.h is).
#pragma once

#include <cstdint>
#include <vector>

#include "st_attn.h"

// Host-resident layout descriptor behind the opaque st_layout_t.
//
// A *segment* is a maximal run of buffer rows whose natural positions are
// consecutive.  Without zigzag the segments are the shards; with zigzag shard
// r contributes two segments (natural chunks r and 2D-1-r, in that order).
struct st_layout {
    int D = 0;
    int zigzag = 0;
    int64_t S = 0;
    std::vector<int64_t> lens;       // D sharding shapes
    std::vector<int64_t> off;        // D+1 prefix offsets
    std::vector<int64_t> seg_buf;    // nseg+1 buffer starts (last = S)
    std::vector<int64_t> seg_nat;    // nseg natural start positions
    std::vector<int> shard_seg;      // D+1: shard r owns segments [shard_seg[r], shard_seg[r+1])
};

namespace st {

constexpr int kMaxSegs = 2 * ST_MAX_SHARDS;

// The layout as kernels see it: a by-value kernel parameter (no device
// allocation), plus the per-segment tile prefix for the launch's tile height.
struct SegTable {
    int32_t nseg;
    int32_t D;
    int32_t S;
    int32_t ntiles;                       // query tiles per (b, h)
    int32_t seg_buf[kMaxSegs + 1];
    int32_t seg_nat[kMaxSegs];
    int32_t seg_tile[kMaxSegs + 1];       // exclusive prefix of tiles per segment
    int32_t shard_seg[ST_MAX_SHARDS + 1];
};

void fill_segtable(const st_layout& L, int tile_rows, SegTable* t);
// The layout of shard r alone, as one rank holds it: D = 1, buffer rows
// 0 .. L_r - 1, the shard's segments with their natural positions.
st_layout shard_layout(const st_layout& L, int r);

// Arguments common to the attention kernels.
struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;            // forward output (input dtype) or nullptr
    float* lse;           // [B,H,S]
    float* part_out;      // partials mode: [D,B,S,H,d] fp32, else nullptr
    float* part_lse;      // partials mode: [D,B,H,S] fp32
    int B, H, d;
    int causal;
    float scale;          // 1/sqrt(d) unless the caller chose another
    int out_dtype;        // dtype of `out`
    // bf16 forward: exact fp16 copy of v scaled by 2^-exps[0] (workspace)
    void* v16;
    unsigned* amax_bits;
    int* exps;
    // ring step: the running state (fp32 [B,Sq,H,d] and [B,H,Sq]) that this
    // call's partial is merged into by the log-sum-exp rule, or nullptr
    const float* prev_out;
    const float* prev_lse;
    // heads h0 .. h0 + hn - 1 only (hn = 0: all heads); the tensors keep all H
    int h0 = 0;
    int hn = 0;
};

// Workspace of st_attn_fwd: bf16 needs the fp16 copy of v plus 256 bytes.
size_t fwd_workspace_bytes(int64_t rows, int d, int dtype);
// Records a CUDA error code for st_last_cuda_error and returns ST_ERR_CUDA (0 -> ST_OK).
int record_cuda_error(int err);
// Argument checks shared by the entry points: 16-byte alignment, and whether a
// pointer addresses device (or managed) memory (NULL passes; host-only query).
bool aligned16(const void* p);
bool on_device(const void* p);

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* out;
    const float* lse;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    float* dq_acc;        // [B,S,H,d] fp32 accumulator (dq itself for fp32 gradients)
    float* delta;         // [B,H,S] fp32 workspace
    int B, H, d;
    int causal;
    float scale;
    int grad_dtype;       // dtype of dq, dk, dv
    int out_dtype;        // dtype of out
    // fp32 inputs: row statistics recomputed in double
    double* lse_d;        // [B,H,S]
    double* delta_d;      // [B,H,S]
    // bf16 inputs: exact fp16 copies of q, k, v, dO scaled by powers of two
    void* h16[4];         // q, k, v, dO as fp16, [B,S,H,d]
    unsigned* amax_bits;  // [4] max |x| of q, k, v, dO (float bits)
    int* exps;            // [8] scale exponents: q, k, v, dO, dS
    int accum;            // ring step: add dK, dV into the fp32 dk, dv instead of writing them
};

// Workspace layout of st_attn_bwd (each piece 256-byte aligned).
struct BwdWorkspace {
    size_t dq_acc, delta, stats, h16, scales, total;
};
BwdWorkspace bwd_workspace_layout(int64_t rows, int d, int dtype);

// ---- launchers (return a cudaError_t value; 0 = success) ----
int launch_fwd_simt(const SegTable& t, const AttnArgs& a, int dtype, void* stream);
// Query tiles [t0, t1) of the layout's 256-row tiles (t1 < 0: all of them).
int launch_fwd_tc(const st_layout& L, const AttnArgs& a, void* stream, bool* handled, int t0 = 0, int t1 = -1);
// Ring step: the query rows of layout Lq (q, out, lse) against the keys of
// layout Lkv (k, v); the two may be different shards held as separate buffers.
int launch_fwd_tc2(const st_layout& Lq, const st_layout& Lkv, const AttnArgs& a, void* stream, int t0 = 0,
                   int t1 = -1);
int fwd_tc_tile_rows();
int launch_bwd_simt(const SegTable& t, const BwdArgs& a, int dtype, void* stream);
int launch_bwd_tc(const st_layout& L, const BwdArgs& a, void* stream, bool* handled);
int launch_bwd_tc2(const st_layout& Lq, const st_layout& Lkv, const BwdArgs& a, void* stream);
// Device error word of the tensor-core kernels (1 after a bounded wait gave
// up, -1 if it could not be read); clear resets it.
int fwd_tc_device_error(bool clear);
int bwd_tc_device_error(bool clear);
int gemm_tc_device_error(bool clear);
int conv_tc_device_error(bool clear);
int selftest_device_error(bool clear);
// C[M, N] = A[M, K] W[N, K]^T on the tensor cores (bf16 in, fp32 accumulation)
int launch_gemm_tc(int M, int N, int K, const void* a, const void* w, void* c, int out_dtype, void* stream);
// halo exchange and sharded 2-D convolution (conv_tc.cu)
int launch_halo_exchange(int D, const int64_t* rows, int W, int C, int h, void* const* shards, void* stream);
int launch_conv_tc(int D, const int64_t* rows, int W, int C_in, int C_out, int k, void* const* in_shards,
                   const void* weight, const float* bias, void* const* out_shards, int out_dtype, void* stream);
// group normalisation of a row-sharded image (norm.cu)
constexpr int kGnStatBlocks = 2048;   // most statistics blocks (sizes the workspace)
size_t group_norm_workspace_bytes(int G);
int launch_group_norm(int D, const int64_t* rows, int W, int C, int G, float eps, const void* const* in,
                      const float* gamma, const float* beta, void* const* out, int out_pad, int out_dtype,
                      void* workspace, void* stream);
// h[M, F] = silu(a w1^T) * (a w3^T), bf16 (gemm_tc.cu)
int launch_gemm_gated(int M, int F, int K, const void* a, const void* w1, const void* w3, void* h, void* stream);
int launch_merge(int D, int B, int H, int64_t S, int d, const float* part_out,
                 const float* part_lse, void* out, float* lse, int out_dtype, void* stream);
int launch_bwd_preprocess(const BwdArgs& a, int64_t S, int dtype, void* stream);
// fp32 inputs: lse and Delta of every row recomputed in double
int launch_rowstats_f64(const SegTable& t, const BwdArgs& a, void* stream);
// bf16 inputs: max |x| and the scaled fp16 copies of q, k, v, dO (q, dO of
// Sq rows, k, v of Skv rows)
int launch_fp16_copies(const BwdArgs& a, int64_t S, void* stream, int64_t Skv = -1);
// One bf16 tensor -> exact fp16 copy scaled by 2^-exps[0] (forward: V)
int launch_fp16_copy1(const void* src, void* dst, int64_t elems, unsigned* amax_bits, int* exps,
                      void* stream);
// The same over a strided set of rows: nrows rows of row8 8-element units each,
// pitch8 units apart (the heads of one group of a [B,S,H,d] tensor); the
// scale and exponent cover these rows only.
int launch_fp16_copy_rows(const void* src, void* dst, int64_t nrows, int row8, int64_t pitch8,
                          unsigned* amax_bits, int* exps, void* stream);
int launch_dq_convert(const BwdArgs& a, int64_t S, int dtype, void* stream);
int launch_permute(const SegTable& t, int B, int H, int d, int dtype, int to_natural,
                   const void* in, void* out, void* stream);

}  // namespace st
