/*
 * st_attn.h -- sharded ring attention on one GPU (GB300, sm_103a).
 *
 * Attention over a sequence that is split into D shards of arbitrary lengths
 * ("sharding shapes": ShardTensor summary, section 2, a fourth metadata item
 * giving each rank's local chunk shape along the sharded axis), computed the
 * ring-attention way (ShardTensor summary, section 4, ring attention): every
 * query shard meets every KV shard in turn and the partial results are merged
 * with the log-sum-exp rule.  An optional zigzag re-partition (TSP summary,
 * "Folding Tensor and Sequence Parallelism", section 2, attention layer) cuts
 * the sequence into 2D chunks and gives rank r chunks r and 2D-1-r so causal
 * work is balanced.
 *
 * On one GPU the D shards are row ranges of one HBM buffer and the "ring" is
 * the kernel's loop over KV shards: no collectives are involved.
 *
 * Conventions shared by every call:
 *   - Tensors q, k, v, out, dout, dq, dk, dv are BSHD: [B, S, H, d], row-major
 *     and contiguous, in *buffer order*: shard 0's rows, then shard 1's, ...
 *     With zigzag, shard r's slab is [chunk r ; chunk 2D-1-r] (natural order
 *     chunk lengths c_r = c_{2D-1-r} = L_r / 2).
 *   - lse is [B, H, S] fp32, natural logarithm of sum_j exp(scale * q.k_j).
 *   - "causal" masks by *natural* sequence position: query i sees key j iff
 *     pos(j) <= pos(i).  Without causal every query sees every key.
 *   - scale <= 0 selects 1/sqrt(d).
 *   - dtype: ST_DTYPE_F32 (fp32 in and out, fp32 SIMT arithmetic) or
 *     ST_DTYPE_BF16 (bf16 in and out, tensor cores, fp32 accumulation).
 *     lse and all accumulators are fp32.
 *   - d (head_dim) is 64 or 128.
 *   - Pointers named q, k, ... are DEVICE pointers that the caller owns and
 *     keeps alive until the work on `stream` has finished; they must be
 *     16-byte aligned.  `stream` is a cudaStream_t (NULL = legacy default
 *     stream).  All GPU work is asynchronous on that stream.  After every
 *     other check, each call asks the CUDA runtime whether its device
 *     pointers address device (or managed) memory and returns
 *     ST_ERR_NOT_DEVICE if one does not, before anything is launched.
 *   - No call allocates device memory.  Scratch that a call needs is a
 *     caller-provided workspace whose size st_attn_workspace_size reports.
 *   - Every call returns ST_OK (0) or a negative ST_ERR_* code; no call aborts
 *     the process or traps the GPU.  On ST_ERR_CUDA, st_last_cuda_error()
 *     returns the CUDA runtime error code that caused it.
 */
#ifndef ST_ATTN_H
#define ST_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    ST_OK = 0,
    ST_ERR_NULL = -1,            /* a required pointer is NULL                      */
    ST_ERR_INVALID_LAYOUT = -2,  /* D out of range, a length < 1, odd zigzag length */
    ST_ERR_UNSUPPORTED = -3,     /* head_dim or dtype not supported                 */
    ST_ERR_MISALIGNED = -4,      /* a tensor pointer is not 16-byte aligned         */
    ST_ERR_WORKSPACE = -5,       /* workspace NULL or smaller than required         */
    ST_ERR_CUDA = -6,            /* a CUDA runtime call or launch failed            */
    ST_ERR_DEVICE_TIMEOUT = -7,  /* a bounded device-side wait gave up              */
    ST_ERR_INVALID_ARG = -8,     /* B, H, S, D or another size is out of range      */
    ST_ERR_SCRATCH_LIMIT = -9,   /* problem too large for st_attn_fwd_noalloc       */
    ST_ERR_NOT_DEVICE = -10      /* a device-pointer argument is not device memory  */
};

enum { ST_DTYPE_F32 = 0, ST_DTYPE_BF16 = 1 };

enum { ST_MAX_SHARDS = 32 };
enum { ST_CONV_MAX_SHARDS = 16 };   /* shards of st_halo_exchange / st_conv2d_sharded */

/* Opaque, host-resident shard-layout descriptor.  Thread-safe to read from
 * several host threads at once; create and destroy are not synchronised. */
typedef struct st_layout st_layout_t;

/* Build a layout from the sharding shapes (ShardTensor summary, section 2).
 *   shard_lens : host array of D lengths L_0..L_{D-1}, each >= 1 (even when
 *                zigzag != 0).  S = sum L_r must be < 2^31.
 *   D          : 1 .. ST_MAX_SHARDS.
 *   zigzag     : 0 = contiguous shards; 1 = zigzag re-partition (TSP summary,
 *                section 2): rank r holds natural chunks r and 2D-1-r.
 *   out        : receives a new descriptor owned by the caller
 *                (free it with st_layout_destroy).
 * Errors: ST_ERR_NULL, ST_ERR_INVALID_LAYOUT.  Host only; no CUDA calls. */
int st_layout_create(const int64_t* shard_lens, int D, int zigzag, st_layout_t** out);

/* Free a descriptor from st_layout_create.  NULL is accepted. */
int st_layout_destroy(st_layout_t* layout);

/* Read back the layout (host arrays, any of them may be NULL):
 *   S       : total rows.
 *   offsets : D+1 prefix offsets, offsets[r] = first buffer row of shard r.
 *   pos     : S natural positions, pos[t] = sequence position of buffer row t.
 *   D, zigzag : the creation arguments. */
int st_layout_query(const st_layout_t* layout, int64_t* S, int64_t* offsets, int64_t* pos,
                    int* D, int* zigzag);

/* Workspace bytes needed by st_attn_fwd (pass = 0) or st_attn_bwd (pass = 1)
 * for these sizes.  The forward needs an fp16 copy of v [B,S,H,d] for bf16
 * inputs and nothing for fp32 (the merge is fused).  The
 * backward needs an fp32 dQ accumulator [B,S,H,d] and the row sums Delta
 * [B,H,S]; bf16 adds four fp16 operand copies [B,S,H,d], fp32 adds the row
 * statistics in double [2,B,H,S]. */
int st_attn_workspace_size(const st_layout_t* layout, int B, int H, int d, int dtype,
                           int pass, size_t* bytes);

/* Forward: out = softmax(scale * Q K^T, masked) V and lse, ring order.
 * Each query tile visits KV shards r, r-1, ..., r+1 (mod D) where r is its
 * own shard -- the order in which rank r receives K/V around a ring -- and
 * folds every KV tile into a running (max, sum, O) state, which is the
 * log-sum-exp merge of the per-shard partials carried out incrementally.
 *   q, k, v   : [B,S,H,d] input dtype.
 *   out_dtype : dtype of out: the input dtype, or ST_DTYPE_F32 (the fp32
 *               accumulator normalised, without a final rounding to bf16).
 *   out       : [B,S,H,d] out_dtype;  lse : [B,H,S] fp32 (may not be NULL).
 *   workspace : st_attn_workspace_size(pass=0) bytes of device memory,
 *               16-byte aligned (bf16: the P V product runs in fp16 on an
 *               exact copy of v scaled by a power of two, made here; fp32:
 *               none, may be NULL / 0).
 * Errors: ST_ERR_NULL, ST_ERR_UNSUPPORTED, ST_ERR_MISALIGNED,
 *         ST_ERR_WORKSPACE, ST_ERR_INVALID_ARG, ST_ERR_CUDA. */
int st_attn_fwd(const st_layout_t* layout, int B, int H, int d, int dtype, int causal,
                float scale, const void* q, const void* k, const void* v, int out_dtype,
                void* out, float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Forward from host buffers, with the copies overlapped with the compute.
 * It computes what st_attn_fwd computes (bf16 in, bf16 out) for inputs and
 * outputs in host memory, and the outputs are bit for bit the same.
 *   q_host, k_host, v_host : host [B,S,H,d] bf16 (page-locked memory lets
 *                            the copies overlap the compute).
 *   out_host : host [B,S,H,d] bf16;  lse_host : host [B,H,S] fp32.
 *   q, k, v, out, lse      : device buffers of the same shapes, owned by
 *                            the caller, used as the staging copies.
 *   workspace, ws_bytes    : as st_attn_fwd (pass 0).
 *   copy_stream            : a second stream, distinct from `stream`, that
 *                            carries the copies.
 * Order of work (stream-ordered: nothing starts before the work already
 * queued on `stream` at the call, which the other streams are made to wait
 * for).  Every query tile needs all of its head's K and V, so the work is
 * split by heads where it can be:
 *   - Head groups, when H has a divisor G (2 <= G <= 16) whose groups of
 *     hn = H / G heads still launch at least four waves of CTAs (the largest
 *     such G), or, for H >= 4 without one, when the whole problem spans eight
 *     waves or more (hn: the fewest heads that make four waves, at least
 *     (H - 2) / 16): a single head first and last, groups of up to hn heads
 *     between.
 *     Per group, V, K and Q of its heads are copied in on copy_stream (2-D
 *     copies, pitch H * d); the fp16 copy of its V (with a scale of its own)
 *     and its attention launch run once they have landed, on `stream` and on
 *     a second stream made for the call, alternately, so that one group's
 *     last wave overlaps the next group's first; its output and lse go back
 *     on copy_stream while the next group computes.  Only the first group's
 *     inputs stand before the first launch, and only the last group's outputs
 *     are copied back after the last.
 *   - Otherwise: V, then K, are copied in whole on copy_stream (the fp16 copy
 *     of V runs on `stream` while K arrives); Q follows in three chunks of
 *     query tiles (a short first chunk of about two waves of CTAs, the bulk,
 *     a short last chunk); each chunk is computed on `stream` once its rows
 *     have arrived, and its output rows and lse go back on copy_stream while
 *     the next chunk computes.
 * When `stream` has completed, every output is in host memory.  A few CUDA
 * events (and, with head groups, one stream) are created and released per
 * call; no device memory is allocated.
 * Errors: as st_attn_fwd, plus ST_ERR_UNSUPPORTED for dtype other than bf16
 * and ST_ERR_INVALID_ARG when copy_stream is NULL or equal to stream. */
int st_attn_fwd_host(const st_layout_t* layout, int B, int H, int d, int dtype, int causal, float scale,
                     const void* q_host, const void* k_host, const void* v_host, void* out_host, float* lse_host,
                     void* q, void* k, void* v, void* out, float* lse, void* workspace, size_t ws_bytes,
                     void* stream, void* copy_stream);

/* Forward for callers that cannot allocate device memory.  No passage of the
 * paper corresponds to it: it is an interface for callers that are handed
 * only their input and output buffers (an operator running inside another
 * runtime), whose memory is fixed at start-up (real-time or certified loops
 * that forbid allocation afterwards), or whose critical path must not call a
 * device allocator (allocations can synchronise and can fail).
 * It computes exactly what st_attn_fwd computes, but the workspace is a
 * fixed 32 MiB array of device memory inside this library instead of a
 * caller buffer:
 *   - every GPU that loads the library holds the array until the process
 *     exits; nothing is allocated or freed per call;
 *   - problems whose workspace (st_attn_workspace_size, pass 0) exceeds
 *     32 MiB are refused with ST_ERR_SCRATCH_LIMIT before anything runs
 *     (bf16: B * S * H * d must stay below about 16.7 million);
 *   - every call looks up the array's device address in the current
 *     device's context (a host-side query that allocates nothing); the first
 *     call on a device may also load the library's device code there, so
 *     make that first call before any stream capture;
 *   - every call on a device uses the same array, so calls whose GPU work
 *     overlaps (on different streams, or from different host threads) race
 *     and must be ordered by the caller.  The array keeps the last call's
 *     contents; whatever a call needs zeroed, it zeroes itself.
 * Other arguments, layouts and errors: as st_attn_fwd (no workspace). */
int st_attn_fwd_noalloc(const st_layout_t* layout, int B, int H, int d, int dtype, int causal,
                        float scale, const void* q, const void* k, const void* v, int out_dtype,
                        void* out, float* lse, void* stream);

/* Forward that stops short of the merge (ShardTensor summary, section 4,
 * ring attention: each query shard meets every KV shard and the partial
 * results are combined): for every query row and every KV shard j it writes
 * the partial (O_j normalised by its own sum, lse_j) over the keys of shard j
 * only -- what each ring step hands to the merge.  A partial with no visible
 * key has O_j = 0 and lse_j = -inf.
 *   partial_out : [D,B,S,H,d] fp32;  partial_lse : [D,B,H,S] fp32.
 *   workspace   : as st_attn_fwd (pass 0): bf16 inputs run the tensor-core
 *                 forward, which restarts its running state at every KV
 *                 shard and writes it out; fp32 needs none (NULL / 0).
 * st_attn_merge of these partials equals st_attn_fwd up to rounding.
 * Errors: as st_attn_fwd. */
int st_attn_fwd_partials(const st_layout_t* layout, int B, int H, int d, int dtype,
                         int causal, float scale, const void* q, const void* k,
                         const void* v, float* partial_out, float* partial_lse,
                         void* workspace, size_t ws_bytes, void* stream);

/* Log-sum-exp merge of D partials (the ring-attention combine step):
 *   L = log sum_j exp(lse_j);  out = sum_j exp(lse_j - L) O_j.
 * All-(-inf) rows give L = -inf and out = 0.
 *   partial_out : [D,B,S,H,d] fp32;  partial_lse : [D,B,H,S] fp32;
 *   out : [B,S,H,d] out_dtype;  lse : [B,H,S] fp32.   d in {64, 128}. */
int st_attn_merge(int D, int B, int H, int64_t S, int d, const float* partial_out,
                  const float* partial_lse, void* out, float* lse, int out_dtype,
                  void* stream);

/* Backward of st_attn_fwd: given out and lse saved by the forward and the
 * output gradient dout, writes dq, dk, dv ([B,S,H,d], all three in grad_dtype).
 * With P = exp(scale*QK^T - lse): dV = P^T dO; dP = dO V^T;
 * Delta = rowsum(dO * out); dS = P * (dP - Delta); dQ = scale dS K;
 * dK = scale dS^T Q.  The KV tiles of shard j meet the query shards in ring
 * order j, j+1, ..., j-1 (mod D).
 *   q, k, v, dout : input dtype;  lse : [B,H,S] fp32 from the forward.
 *   out, out_dtype : the forward output, in the input dtype or ST_DTYPE_F32
 *                (an fp32 out gives Delta without the bf16 rounding of out).
 *   grad_dtype : ST_DTYPE_F32 (fp32 gradients, no final rounding) or the
 *                input dtype.
 *   workspace  : at least st_attn_workspace_size(pass=1) bytes of device
 *                memory, 16-byte aligned; its contents on entry do not matter.
 * bf16 inputs run on tcgen05 tensor cores with fp16 operands (exact copies
 * of q, k, v, dO scaled by powers of two, made in the workspace) so that P
 * and dS carry 11 significant bits; fp32 inputs run on the SIMT path with the
 * row statistics (lse, Delta) recomputed in double.
 * Errors: as st_attn_fwd, plus ST_ERR_WORKSPACE. */
int st_attn_bwd(const st_layout_t* layout, int B, int H, int d, int dtype, int causal,
                float scale, const void* q, const void* k, const void* v,
                const void* out, int out_dtype, const float* lse, const void* dout,
                int grad_dtype, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                void* stream);

/*
 * Ring attention across ranks (ShardTensor summary, section 4, ring
 * attention; TSP summary, section 2, attention layer, for the zigzag
 * re-partition).  Rank r keeps the query rows of shard r of the layout; the
 * K/V shards travel round a ring of ranks, so that at step t = 0 .. D-1 rank
 * r holds the K/V of shard (r - t) mod D -- its own at step 0, then each step
 * the block its left neighbour held -- and folds that shard's partial result
 * into its running result by the log-sum-exp rule.  In training the K/V
 * shards travel with fp32 dK/dV accumulators, to which every rank adds its
 * queries' contributions, and one more hop after the last step brings them to
 * the shard's owner.  The causal mask follows the natural positions of both
 * shards.  Only bf16 inputs (the tensor-core path); a shard's tensors are
 * [B, L_r, H, d] (q, k, v, out, dout) and [B, H, L_r] (lse), contiguous, in the
 * rank's buffer order (with zigzag, chunk r then chunk 2D-1-r).
 */

/* Workspace bytes for any pair of shards of the layout (sized by the longest
 * shard): which = 0 st_ring_fwd_step, 1 st_ring_bwd_step, 2 st_ring_fwd_local,
 * 3 st_ring_bwd_local. */
int st_ring_workspace_size(const st_layout_t* layout, int B, int H, int d, int which, size_t* bytes);

/* One forward step of rank q_shard: its query rows q against the K/V block of
 * shard kv_shard that it holds at this step.  With prev_out / prev_lse NULL
 * (the first step) out, lse = this block's partial (O normalised by its own
 * sum, lse = log of that sum; no visible key: O = 0, lse = -inf); otherwise
 * the partial is merged with the running state (prev_out fp32 [B,L_q,H,d],
 * prev_lse [B,H,L_q]) into out, lse:  L = log(e^lse_prev + e^lse_blk),
 * out = e^(lse_prev - L) prev_out + e^(lse_blk - L) O_blk.  out and lse may
 * alias prev_out and prev_lse (fp32 out).
 *   q        : [B, L_q, H, d] bf16;  k, v : [B, L_kv, H, d] bf16.
 *   out_dtype: ST_DTYPE_F32 (the running state) or ST_DTYPE_BF16 (a last step).
 *   dtype    : ST_DTYPE_BF16.
 *   workspace: st_ring_workspace_size(which = 0) bytes of device memory.
 * One fp16 copy of v and the fused kernel on `stream`.
 * Errors: as st_attn_fwd, plus ST_ERR_INVALID_ARG for a shard index out of
 * range and ST_ERR_NULL when only one of prev_out, prev_lse is given. */
int st_ring_fwd_step(const st_layout_t* layout, int q_shard, int kv_shard, int B, int H, int d, int dtype,
                     int causal, float scale, const void* q, const void* k, const void* v,
                     const float* prev_out, const float* prev_lse, int out_dtype, void* out, float* lse,
                     void* workspace, size_t ws_bytes, void* stream);

/* One backward step of rank q_shard holding shard kv_shard's K/V and their
 * travelling gradient accumulators: adds this block's contributions
 *   dV_kv += P^T dO,  dK_kv += scale dS^T Q,  dQ_q += scale dS K
 * (P = exp(scale QK^T - lse), dS = P o (dO V^T - Delta), Delta = rowsum(dO o
 * out)) to the fp32 dk, dv [B,L_kv,H,d] and dq [B,L_q,H,d].  first_q = 1
 * zeroes dq first (the rank's first step).  out: the rank's forward output
 * (bf16 or fp32, out_dtype), lse its fp32 lse.  dtype: ST_DTYPE_BF16.
 * workspace: st_ring_workspace_size(which = 1) bytes.
 * Errors: as st_attn_bwd, plus ST_ERR_INVALID_ARG for a shard index out of
 * range. */
int st_ring_bwd_step(const st_layout_t* layout, int q_shard, int kv_shard, int B, int H, int d, int dtype,
                     int causal, float scale, const void* q, const void* k, const void* v, const void* out,
                     int out_dtype, const float* lse, const void* dout, int first_q, float* dq, float* dk,
                     float* dv, void* workspace, size_t ws_bytes, void* stream);

/* The whole ring forward with the D ranks held on this one GPU: host arrays of
 * D device pointers give rank r's q, k, v (its shard) and its outputs out
 * ([B,L_r,H,d], out_dtype) and lse ([B,H,L_r]).  The K/V blocks pass from
 * rank to rank by device-to-device copies on copy_stream (a stream other than
 * `stream`) into two receive buffers per rank in the workspace, each step's
 * copies running while the previous blocks are computed on `stream`.  When
 * `stream` completes, every rank's out and lse hold its queries' attention
 * over the whole sequence.  workspace: st_ring_workspace_size(which = 2).
 * Errors: as st_ring_fwd_step, plus ST_ERR_INVALID_ARG when copy_stream is
 * NULL or equal to stream. */
int st_ring_fwd_local(const st_layout_t* layout, int B, int H, int d, int causal, float scale,
                      const void* const* q, const void* const* k, const void* const* v, int out_dtype,
                      void* const* out, float* const* lse, void* workspace, size_t ws_bytes, void* stream,
                      void* copy_stream);

/* The whole ring backward with the D ranks on this one GPU: rank r's q, k, v,
 * out (out_dtype), lse, dout in, fp32 dq, dk, dv of its shard out.  K and V
 * pass on while a step computes; the dK/dV accumulators pass on after it has
 * added to them, and after the last step they reach their owner's dk, dv.
 * workspace: st_ring_workspace_size(which = 3).  Errors: as
 * st_ring_bwd_step, plus ST_ERR_INVALID_ARG for copy_stream. */
int st_ring_bwd_local(const st_layout_t* layout, int B, int H, int d, int causal, float scale,
                      const void* const* q, const void* const* k, const void* const* v, const void* const* out,
                      int out_dtype, const float* const* lse, const void* const* dout, float* const* dq,
                      float* const* dk, float* const* dv, void* workspace, size_t ws_bytes, void* stream,
                      void* copy_stream);

/* Backward preprocess on its own: Delta[b,h,i] = sum_c dout[b,i,h,c] *
 * out[b,i,h,c] in fp32 -- the row sums of dO o O that the backward subtracts
 * from dP (the gradient of the softmax).  A ring backward computes them once
 * per rank, before its steps.
 *   out  : [B,S,H,d] in out_dtype (dtype or ST_DTYPE_F32);  dout : [B,S,H,d]
 *   dtype;  delta : [B,H,S] fp32.  One launch, HBM-bound.
 * Errors: ST_ERR_NULL, ST_ERR_INVALID_ARG, ST_ERR_UNSUPPORTED,
 * ST_ERR_MISALIGNED, ST_ERR_NOT_DEVICE, ST_ERR_CUDA. */
int st_attn_bwd_delta(int B, int H, int64_t S, int d, int dtype, const void* out, int out_dtype,
                      const void* dout, float* delta, void* stream);

/* fp32 accumulator -> dst_dtype (ST_DTYPE_BF16: rounded to nearest even;
 * ST_DTYPE_F32: copied): n elements, the conversion the backward applies to
 * its dQ accumulator, also the last step of an fp32 ring result.  One
 * launch, HBM-bound.  Errors: ST_ERR_NULL, ST_ERR_INVALID_ARG,
 * ST_ERR_UNSUPPORTED, ST_ERR_MISALIGNED, ST_ERR_NOT_DEVICE, ST_ERR_CUDA. */
int st_convert_f32(int64_t n, const float* src, void* dst, int dst_dtype, void* stream);

/* The exact fp16 operand copy the tensor-core kernels run on: dst = src *
 * 2^-e in fp16 for n bf16 values (n a multiple of 8), e chosen from max|src|
 * so that max|src| * 2^-e lies in [2^13, 2^14) -- bf16's 8 significant bits
 * fit in fp16's 11, so every value within 2^-27 of the maximum is copied
 * exactly.  exps[0] receives e (device int); scratch: 16 device bytes for the
 * maximum.  Two launches (max, copy), HBM-bound.
 * Errors: ST_ERR_NULL, ST_ERR_INVALID_ARG, ST_ERR_MISALIGNED,
 * ST_ERR_NOT_DEVICE, ST_ERR_CUDA. */
int st_fp16_scaled_copy(int64_t n, const void* src, void* dst, int* exps, void* scratch, void* stream);

/* Reorder rows between buffer order and natural sequence order:
 *   to_natural = 1 : out[:, pos(t)] = in[:, t]   (buffer -> natural)
 *   to_natural = 0 : out[:, t] = in[:, pos(t)]   (natural -> buffer)
 * in/out : [B,S,H,d] dtype, distinct buffers. */
int st_permute(const st_layout_t* layout, int B, int H, int d, int dtype, int to_natural,
               const void* in, void* out, void* stream);

/*
 * Projection GEMM:  y[M, N] = x[M, K] w[N, K]^T.
 *
 * The projections on either side of the attention (TSP summary, "Folding
 * Tensor and Sequence Parallelism", section 2, attention layer, broadcast
 * schedule: every rank computes the local projections of its sequence shard
 * with each packed W_Q, W_K, W_V, W_O weight shard in turn).  On one GPU the
 * sequence shards are row ranges of x (in buffer order) and the weight shards
 * row ranges of w, so every (sequence shard, weight shard) product is a block
 * of this one product: for the input projections x is [B*S, hidden] and w the
 * packed [3*H*d, hidden] W_Q|W_K|W_V, whose output viewed as [B, S, 3, H, d]
 * holds q, k and v; for the output projection x is the attention output
 * [B*S, H*d] and w is W_O [hidden, H*d].
 *
 *   x   : device, bf16, [M, K] row-major.
 *   w   : device, bf16, [N, K] row-major (a Linear layer's [out, in] weight).
 *   y   : device, [M, N] row-major, out_dtype ST_DTYPE_BF16 or ST_DTYPE_F32.
 *   Tensor cores with fp32 accumulation over K.  N and K must be multiples of
 *   8 (16-byte rows for the TMA), pointers 16-byte aligned.
 *
 * Returns ST_ERR_NULL, ST_ERR_INVALID_ARG (sizes), ST_ERR_UNSUPPORTED (dtype),
 * ST_ERR_MISALIGNED or ST_ERR_CUDA.  The caller owns every buffer; nothing is
 * allocated.
 */
int st_proj_gemm(int M, int N, int K, const void* x, const void* w, void* y, int out_dtype,
                 void* stream);

/*
 * Gated MLP:  h = silu(x W1^T) * (x W3^T),  y = h W2^T,  silu(a) = a / (1 + e^-a).
 *
 * The feed-forward layer that TSP pairs with its ring schedule (TSP summary,
 * "Folding Tensor and Sequence Parallelism", section 2, gated MLP layer: the
 * W1, W2, W3 shards travel round the ring while each rank keeps its tokens
 * and adds up its partial outputs, so no all-reduce is needed).  A weight
 * shard j is a range F_j of hidden units: rows F_j of W1 and W3 and columns
 * F_j of W2.  The partial output of shard j is silu(x W1_j^T) * (x W3_j^T)
 * W2_j^T, and the partials over all shards sum to the product above.  On one
 * GPU every shard is resident, so the sum over shards is the K loop of the
 * second GEMM, over all F hidden units.
 *
 *   x   : device, bf16, [M, hidden] row-major (M tokens in buffer order).
 *   w1  : device, bf16, [F, hidden] (gate weight, a Linear layer's [out, in]).
 *   w3  : device, bf16, [F, hidden] (up weight).
 *   w2  : device, bf16, [hidden, F] (down weight).
 *   h   : device, bf16, [M, F]: caller-owned workspace; holds the gated
 *         activation on return (rounded once to bf16 from fp32 accumulators,
 *         then the A operand of the down projection).
 *   y   : device, [M, hidden], out_dtype ST_DTYPE_BF16 or ST_DTYPE_F32.
 *   hidden and F must be multiples of 8, pointers 16-byte aligned.  Two
 *   tensor-core launches on `stream`; fp32 accumulation in both.
 *
 * Returns ST_ERR_NULL, ST_ERR_INVALID_ARG (sizes), ST_ERR_UNSUPPORTED (dtype),
 * ST_ERR_MISALIGNED or ST_ERR_CUDA.  Nothing is allocated.
 */
int st_gated_mlp(int M, int hidden, int F, const void* x, const void* w1, const void* w3, const void* w2,
                 void* h, void* y, int out_dtype, void* stream);

/*
 * Halo exchange of a row-sharded image.
 *
 * ShardTensor summary, "ShardTensor" section 2, implementation details,
 * communication: a convolution or normalisation over a spatially sharded
 * input needs the neighbouring pixels held by the adjacent chunks (the
 * "halo").  The H image rows are split into D shards of rows[r] >= 1 rows
 * (uneven sharding shapes, section 2), in order.  Shard r is its own buffer,
 * as it would be on its own device.
 *
 *   rows   : host, D values; the image has H = sum(rows) rows.
 *   shards : host array of D device pointers.  shards[r] is bf16
 *            [rows[r] + 2*halo, W, C] (channels last).  Its rows
 *            halo .. halo + rows[r] - 1 hold image rows off_r .. off_r + rows[r] - 1,
 *            where off_r = rows[0] + ... + rows[r-1].
 *   Fills, in place, the halo rows above and below each shard's own rows with
 *   the image rows off_r - halo .. off_r - 1 and off_r + rows[r] ..
 *   off_r + rows[r] + halo - 1, taken from whichever shards own them (a shard
 *   shorter than halo passes on rows of shards further away).  Rows outside
 *   the image are written as zeros.  Only pad rows are written, only own rows
 *   read.
 *   1 <= D <= ST_CONV_MAX_SHARDS, 0 <= halo <= 3, C a multiple of 8,
 *   W*C <= 2^24, H <= 2^24; pointers 16-byte aligned.  One launch on `stream`.
 *
 * Returns ST_ERR_NULL, ST_ERR_INVALID_LAYOUT (a shard of < 1 row),
 * ST_ERR_INVALID_ARG, ST_ERR_MISALIGNED or ST_ERR_CUDA.  Nothing is allocated.
 */
int st_halo_exchange(int D, const int64_t* rows, int W, int C, int halo, void* const* shards, void* stream);

/*
 * 2-D convolution of a row-sharded image, from halo-padded shards.
 *
 *   y_r[i, j, o] = bias[o] + sum_{u,v,c} xpad_r[i + u, j + v - h, c] * w[o, u, v, c]
 *
 * Here h = (k - 1) / 2. xpad_r is shard r padded with h rows on each side, as
 * st_halo_exchange leaves it, and it is zero outside 0 <= j + v - h < W.
 * After the exchange, the shards' outputs stacked in order are the
 * cross-correlation of the whole image: the convolution of deep-learning
 * layers, stride 1, zero padding h, output as large as the input. That is the
 * reading this library takes of the convolution the same passage names.
 *
 *   rows       : host, D shard lengths (as st_halo_exchange).
 *   in_shards  : host array of D device pointers, bf16 [rows[r] + 2h, W, C_in].
 *   weight     : device, bf16 [C_out, k, k, C_in] (channels last).
 *   bias       : device fp32 [C_out], or NULL for none.
 *   out_shards : host array of D device pointers, [rows[r], W, C_out] in
 *                out_dtype (ST_DTYPE_BF16 or ST_DTYPE_F32).
 *   Tensor cores: bf16 products, fp32 accumulation over k*k*C_in.
 *   k odd in 1..7; C_in a multiple of 64 (<= 4096); C_out a multiple of 8
 *   (<= 4096); 1 <= D <= ST_CONV_MAX_SHARDS; pointers 16-byte aligned.  One
 *   launch on `stream`.
 *
 * Returns ST_ERR_NULL, ST_ERR_INVALID_LAYOUT, ST_ERR_INVALID_ARG,
 * ST_ERR_UNSUPPORTED (dtype), ST_ERR_MISALIGNED or ST_ERR_CUDA.  Nothing is
 * allocated.
 */
int st_conv2d_sharded(int D, const int64_t* rows, int W, int C_in, int C_out, int k, void* const* in_shards,
                      const void* weight, const float* bias, void* const* out_shards, int out_dtype,
                      void* stream);

/*
 * Group normalisation of a row-sharded image.
 *
 * ShardTensor summary, "ShardTensor" section 2, implementation details,
 * communication: normalisation over a spatially sharded input needs a
 * collective, here the all-reduce of per-group statistics, to give the
 * numbers of the layer on the whole image.  Group normalisation is the
 * reading this library takes of the normalisation that passage names.
 *
 *   y[i, j, c] = (x[i, j, c] - mu_g) / sqrt(var_g + eps) * gamma[c] + beta[c]
 *
 * Channel c is in group g = c / (C / G).  mu_g and var_g (biased) are taken
 * over every pixel of every shard and every channel of the group.
 *
 *   rows       : host, D shard lengths (image rows), as st_halo_exchange.
 *   in_shards  : host array of D device pointers, bf16 [rows[r], W, C].
 *   gamma, beta: device fp32 [C], or NULL for 1 and 0.
 *   out_shards : host array of D device pointers, [rows[r] + 2*out_pad, W, C]
 *                in out_dtype (ST_DTYPE_BF16 or ST_DTYPE_F32).  Rows
 *                out_pad .. out_pad + rows[r] - 1 are written and the pad rows
 *                left as they are, so the output can go straight into
 *                st_halo_exchange and st_conv2d_sharded (out_pad = (k-1)/2).
 *   workspace  : device, >= st_group_norm_workspace_size bytes, 16-byte
 *                aligned; the per-block statistics and the combined mean and
 *                1/std per group (fp64) are left there.
 *   C a power of two in 8 .. 2048; C a multiple of G; C / G a multiple of 8;
 *   eps > 0; 0 <= out_pad <= 3; 1 <= D <= ST_CONV_MAX_SHARDS.
 *   Statistics are kept in fp32 per thread (shifted sums), merged in fp32
 *   per block and in fp64 across blocks.  Three launches on `stream`.
 *
 * Returns ST_ERR_NULL, ST_ERR_INVALID_LAYOUT, ST_ERR_INVALID_ARG,
 * ST_ERR_UNSUPPORTED (dtype), ST_ERR_MISALIGNED, ST_ERR_WORKSPACE or
 * ST_ERR_CUDA.  Nothing is allocated.
 */
int st_group_norm_workspace_size(int C, int G, size_t* bytes);
int st_group_norm_sharded(int D, const int64_t* rows, int W, int C, int G, float eps, const void* const* in_shards,
                          const float* gamma, const float* beta, void* const* out_shards, int out_pad,
                          int out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Wait for `stream`, then report (and clear) the device error word of the
 * tensor-core kernels: ST_ERR_DEVICE_TIMEOUT if one of their bounded
 * barrier waits gave up since the last call (the kernel then stopped early
 * and its outputs are not valid), else ST_OK.  Blocks the host. */
int st_device_error(void* stream);

/* Self-test of the bounded device waits (failure detection; the paper has no
 * counterpart).  Launches one CTA of one warp on `stream` that initialises an
 * mbarrier nothing ever arrives at and waits on it with the kernels' bounded
 * wait, giving up after limit_cycles clock cycles of polling (1 .. 4e9; the
 * kernels' own limit is 4e9, about 2 s).  No copy, MMA or tensor-memory
 * allocation is in flight, so the kernel only records the timeout in the
 * device error word and returns: st_device_error then reports
 * ST_ERR_DEVICE_TIMEOUT once and clears it, and the context stays usable.
 * Errors: ST_ERR_INVALID_ARG (limit out of range), ST_ERR_CUDA (launch). */
int st_selftest_bounded_wait(long long limit_cycles, void* stream);

/* Human-readable text for a status code (static storage). */
const char* st_error_string(int code);

/* 1 if p addresses device (or managed) memory, the check every entry point
 * applies to its device pointers; 0 for NULL, host memory (page-locked or
 * not) and addresses the runtime does not know.  Host only, never launches. */
int st_is_device_pointer(const void* p);

/* CUDA runtime error code behind the most recent ST_ERR_CUDA of this thread. */
int st_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ST_ATTN_H */
