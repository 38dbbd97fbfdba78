// Ring attention across ranks: one step of a rank, and the whole ring with the
// ranks held on one GPU.
//
// ShardTensor summary, section 4, ring attention: the sequence is split into
// D shards (sharding shapes of any lengths, section 2), rank r keeps the
// queries of shard r, and the K/V shards travel round a ring of ranks -- at
// step t rank r holds the K/V of shard (r - t) mod D, computes that shard's
// partial result for its queries while the next shard is in transit, and
// folds it into its running result by the log-sum-exp rule.  In training the
// K/V shards travel with their dK/dV accumulators, to which every rank adds
// its queries' contributions; after the last step one more hop brings them
// home.  With the TSP zigzag re-partition (TSP summary, section 2, attention
// layer) a shard is two chunks of the sequence, and the causal mask follows
// the natural positions of both.
//
// Per step the work is the tensor-core forward or backward over one (query
// shard, KV shard) block: the kernels take the query rows and the keys as two
// separate layouts, each one shard held in its own buffer, and the forward
// merges its result into the running state in its epilogue.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "common.h"

namespace {

int cuda_status(int err) { return st::record_cuda_error(err); }

using st::aligned16;
using st::on_device;

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

int64_t longest_shard(const st_layout& L) { return *std::max_element(L.lens.begin(), L.lens.end()); }

int check_ring(const st_layout_t* L, int B, int H, int d, int dtype, float* scale) {
    if (!L) return ST_ERR_NULL;
    if (B < 1 || H < 1 || (int64_t)B * H > 65535) return ST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ST_ERR_UNSUPPORTED;
    if (dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;   // the tensor-core path
    if (!std::isfinite(*scale)) return ST_ERR_INVALID_ARG;
    if (*scale <= 0.f) *scale = 1.0f / std::sqrt((float)d);
    return ST_OK;
}

// Workspace of one step, sized for the longest shard: forward -- the fp16
// copy of the KV block's v and its scale; backward -- Delta of the query
// rows, the fp16 copies of q, k, v, dO and their scales.
size_t fwd_step_bytes(const st_layout& L, int B, int H, int d) {
    return st::fwd_workspace_bytes((int64_t)B * longest_shard(L) * H, d, ST_DTYPE_BF16);
}
size_t bwd_step_bytes(const st_layout& L, int B, int H, int d) {
    const int64_t rows = (int64_t)B * longest_shard(L) * H;
    return up256((size_t)rows * 4) + 4 * up256((size_t)rows * d * 2) + 256;
}

// The whole ring on one GPU: per rank two receive buffers of the travelling
// block (K and V; in the backward also the fp32 dK and dV accumulators), and
// in the forward the fp32 running state when the output is bf16.
struct LocalRing {
    size_t blk16, blk32, lse32, per_rank, step, total;
};
LocalRing local_layout(const st_layout& L, int B, int H, int d, int pass) {
    LocalRing w{};
    const int64_t rows = (int64_t)B * longest_shard(L) * H;
    w.blk16 = up256((size_t)rows * d * 2);
    w.blk32 = up256((size_t)rows * d * 4);
    w.lse32 = up256((size_t)rows * 4);
    if (pass == 0)
        w.per_rank = 2 * 2 * w.blk16 + w.blk32 + w.lse32;       // 2 x (K, V), running out + lse
    else
        w.per_rank = 2 * (2 * w.blk16 + 2 * w.blk32);           // 2 x (K, V, dK, dV)
    w.step = pass == 0 ? up256(fwd_step_bytes(L, B, H, d)) : up256(bwd_step_bytes(L, B, H, d));
    w.total = (size_t)L.D * w.per_rank + w.step;
    return w;
}

}  // namespace

extern "C" int st_ring_workspace_size(const st_layout_t* L, int B, int H, int d, int which, size_t* bytes) {
    float scale = 1.f;
    if (!bytes) return ST_ERR_NULL;
    const int rc = check_ring(L, B, H, d, ST_DTYPE_BF16, &scale);
    if (rc != ST_OK) return rc;
    switch (which) {
        case 0: *bytes = fwd_step_bytes(*L, B, H, d); break;
        case 1: *bytes = bwd_step_bytes(*L, B, H, d); break;
        case 2: *bytes = local_layout(*L, B, H, d, 0).total; break;
        case 3: *bytes = local_layout(*L, B, H, d, 1).total; break;
        default: return ST_ERR_INVALID_ARG;
    }
    return ST_OK;
}

extern "C" int st_ring_fwd_step(const st_layout_t* L, int q_shard, int kv_shard, int B, int H, int d, int dtype,
                                int causal, float scale, const void* q, const void* k, const void* v,
                                const float* prev_out, const float* prev_lse, int out_dtype, void* out, float* lse,
                                void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_ring(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (q_shard < 0 || q_shard >= L->D || kv_shard < 0 || kv_shard >= L->D) return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || !lse) return ST_ERR_NULL;
    if ((prev_out == nullptr) != (prev_lse == nullptr)) return ST_ERR_NULL;
    if (!workspace) return ST_ERR_WORKSPACE;
    const void* ptrs[] = {q, k, v, out, lse, prev_out, prev_lse, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return ST_ERR_MISALIGNED;
    const size_t need = fwd_step_bytes(*L, B, H, d);
    if (ws_bytes < need) return ST_ERR_WORKSPACE;
    for (const void* p : ptrs)
        if (!on_device(p)) return ST_ERR_NOT_DEVICE;
    const st_layout Lq = st::shard_layout(*L, q_shard), Lkv = st::shard_layout(*L, kv_shard);
    st::AttnArgs a{q, k, v, out, lse, nullptr, nullptr, B, H, d, causal ? 1 : 0, scale, out_dtype,
                   nullptr, nullptr, nullptr, prev_out, prev_lse};
    char* ws = static_cast<char*>(workspace);
    a.v16 = ws;
    a.amax_bits = reinterpret_cast<unsigned*>(ws + need - 256);
    a.exps = reinterpret_cast<int*>(ws + need - 128);
    rc = cuda_status(st::launch_fp16_copy1(v, a.v16, (int64_t)B * Lkv.S * H * d, a.amax_bits, a.exps, stream));
    if (rc != ST_OK) return rc;
    return cuda_status(st::launch_fwd_tc2(Lq, Lkv, a, stream));
}

namespace {

// One backward step without the argument checks (the callers make them).
int bwd_step(const st_layout& L, int q_shard, int kv_shard, int B, int H, int d, int causal, float scale,
             const void* q, const void* k, const void* v, const void* out, int out_dtype, const float* lse,
             const void* dout, int first_q, float* dq, float* dk, float* dv, void* workspace, void* stream) {
    const st_layout Lq = st::shard_layout(L, q_shard), Lkv = st::shard_layout(L, kv_shard);
    const int64_t rows = (int64_t)B * longest_shard(L) * H;
    char* ws = static_cast<char*>(workspace);
    st::BwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.dout = dout;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dq_acc = dq;
    a.delta = reinterpret_cast<float*>(ws);
    a.B = B;
    a.H = H;
    a.d = d;
    a.causal = causal ? 1 : 0;
    a.scale = scale;
    a.grad_dtype = ST_DTYPE_F32;
    a.out_dtype = out_dtype;
    a.accum = 1;
    size_t off = up256((size_t)rows * 4);
    for (int i = 0; i < 4; ++i) {
        a.h16[i] = ws + off;
        off += up256((size_t)rows * d * 2);
    }
    a.amax_bits = reinterpret_cast<unsigned*>(ws + off);
    a.exps = reinterpret_cast<int*>(ws + off + 64);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int rc;
    if (first_q) {
        rc = cuda_status((int)cudaMemsetAsync(dq, 0, (size_t)B * Lq.S * H * d * sizeof(float), cs));
        if (rc != ST_OK) return rc;
    }
    rc = cuda_status(st::launch_bwd_preprocess(a, Lq.S, ST_DTYPE_BF16, stream));
    if (rc != ST_OK) return rc;
    rc = cuda_status((int)cudaMemsetAsync(a.amax_bits, 0, 64, cs));
    if (rc != ST_OK) return rc;
    rc = cuda_status(st::launch_fp16_copies(a, Lq.S, stream, Lkv.S));
    if (rc != ST_OK) return rc;
    return cuda_status(st::launch_bwd_tc2(Lq, Lkv, a, stream));
}

}  // namespace

extern "C" int st_ring_bwd_step(const st_layout_t* L, int q_shard, int kv_shard, int B, int H, int d, int dtype,
                                int causal, float scale, const void* q, const void* k, const void* v,
                                const void* out, int out_dtype, const float* lse, const void* dout, int first_q,
                                float* dq, float* dk, float* dv, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_ring(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (q_shard < 0 || q_shard >= L->D || kv_shard < 0 || kv_shard >= L->D) return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return ST_ERR_NULL;
    if (!workspace || ws_bytes < bwd_step_bytes(*L, B, H, d)) return ST_ERR_WORKSPACE;
    const void* ptrs[] = {q, k, v, out, lse, dout, dq, dk, dv, workspace};
    for (const void* p : ptrs)
        if (!aligned16(p)) return ST_ERR_MISALIGNED;
    for (const void* p : ptrs)
        if (!on_device(p)) return ST_ERR_NOT_DEVICE;
    return bwd_step(*L, q_shard, kv_shard, B, H, d, causal ? 1 : 0, scale, q, k, v, out, out_dtype, lse, dout,
                    first_q ? 1 : 0, dq, dk, dv, workspace, stream);
}

namespace {

// Events of a local ring: per step, "computed" (on the compute stream) and
// "arrived" (on the copy stream).  Created and released per call.
struct Events {
    std::vector<cudaEvent_t> ev;
    int make(int n) {
        ev.assign(n, nullptr);
        for (auto& e : ev) {
            const int rc = cuda_status((int)cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
            if (rc != ST_OK) return rc;
        }
        return ST_OK;
    }
    ~Events() {
        for (auto& e : ev)
            if (e) cudaEventDestroy(e);   // released once pending work has passed it
    }
};

int check_local(const st_layout_t* L, int B, int H, int d, float* scale, void* workspace, size_t ws_bytes, int pass,
                void* stream, void* copy_stream) {
    int rc = check_ring(L, B, H, d, ST_DTYPE_BF16, scale);
    if (rc != ST_OK) return rc;
    if (!copy_stream || copy_stream == stream) return ST_ERR_INVALID_ARG;
    if (!workspace) return ST_ERR_WORKSPACE;
    if (ws_bytes < local_layout(*L, B, H, d, pass).total) return ST_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
    return ST_OK;
}

template <typename P>
int check_ptr_array(int D, P const* arr) {
    if (!arr) return ST_ERR_NULL;
    for (int r = 0; r < D; ++r) {
        if (!arr[r]) return ST_ERR_NULL;
        if (!aligned16(arr[r])) return ST_ERR_MISALIGNED;
    }
    return ST_OK;
}

template <typename P>
bool ptr_array_on_device(int D, P const* arr) {
    for (int r = 0; r < D; ++r)
        if (!on_device(arr[r])) return false;
    return true;
}

}  // namespace

extern "C" int st_ring_fwd_local(const st_layout_t* L, int B, int H, int d, int causal, float scale,
                                 const void* const* q, const void* const* k, const void* const* v, int out_dtype,
                                 void* const* out, float* const* lse, void* workspace, size_t ws_bytes, void* stream,
                                 void* copy_stream) {
    int rc = check_local(L, B, H, d, &scale, workspace, ws_bytes, 0, stream, copy_stream);
    if (rc != ST_OK) return rc;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    const int D = L->D;
    if ((rc = check_ptr_array(D, q)) || (rc = check_ptr_array(D, k)) || (rc = check_ptr_array(D, v)) ||
        (rc = check_ptr_array(D, out)) || (rc = check_ptr_array(D, lse)))
        return rc;
    if (!ptr_array_on_device(D, q) || !ptr_array_on_device(D, k) || !ptr_array_on_device(D, v) ||
        !ptr_array_on_device(D, out) || !ptr_array_on_device(D, lse) || !on_device(workspace))
        return ST_ERR_NOT_DEVICE;
    const LocalRing w = local_layout(*L, B, H, d, 0);
    char* ws = static_cast<char*>(workspace);
    auto recv_k = [&](int r, int slot) { return ws + r * w.per_rank + slot * 2 * w.blk16; };
    auto recv_v = [&](int r, int slot) { return recv_k(r, slot) + w.blk16; };
    auto run_out = [&](int r) { return reinterpret_cast<float*>(ws + r * w.per_rank + 4 * w.blk16); };
    auto run_lse = [&](int r) { return reinterpret_cast<float*>(ws + r * w.per_rank + 4 * w.blk16 + w.blk32); };
    void* step_ws = ws + (size_t)D * w.per_rank;
    cudaStream_t cs = static_cast<cudaStream_t>(stream), xs = static_cast<cudaStream_t>(copy_stream);
    Events e;
    // ev[0]: entry of `stream`; computed[t] = ev[1 + t]; arrived[t] = ev[1 + D + t]
    if ((rc = e.make(1 + 2 * D)) != ST_OK) return rc;
    auto ck = [](cudaError_t x) { return cuda_status((int)x); };
    // the copies may only start after the work already queued on `stream`
    if ((rc = ck(cudaEventRecord(e.ev[0], cs))) != ST_OK) return rc;
    if ((rc = ck(cudaStreamWaitEvent(xs, e.ev[0], 0))) != ST_OK) return rc;
    const size_t row_bytes = (size_t)H * d * 2;
    // the K/V block rank r holds at step t: its own at t = 0, then a receive buffer
    auto held_k = [&](int r, int t) -> const void* { return t == 0 ? k[r] : recv_k(r, t & 1); };
    auto held_v = [&](int r, int t) -> const void* { return t == 0 ? v[r] : recv_v(r, t & 1); };
    for (int t = 0; t < D; ++t) {
        // transit for step t + 1: every rank passes the block it holds to the
        // next rank, while step t computes; the receive buffer it overwrites was
        // last read by step t - 1
        if (t + 1 < D) {
            if (t >= 1 && (rc = ck(cudaStreamWaitEvent(xs, e.ev[1 + t - 1], 0))) != ST_OK) return rc;
            for (int r = 0; r < D; ++r) {
                const int src = (r + D - 1) % D;
                const int j = ((src - t) % D + D) % D;           // the shard the sender holds
                const size_t n = (size_t)B * L->lens[j] * row_bytes;
                if ((rc = ck(cudaMemcpyAsync(recv_k(r, (t + 1) & 1), held_k(src, t), n, cudaMemcpyDeviceToDevice,
                                             xs))) != ST_OK)
                    return rc;
                if ((rc = ck(cudaMemcpyAsync(recv_v(r, (t + 1) & 1), held_v(src, t), n, cudaMemcpyDeviceToDevice,
                                             xs))) != ST_OK)
                    return rc;
            }
            if ((rc = ck(cudaEventRecord(e.ev[1 + D + t + 1], xs))) != ST_OK) return rc;
        }
        if (t >= 1 && (rc = ck(cudaStreamWaitEvent(cs, e.ev[1 + D + t], 0))) != ST_OK) return rc;
        for (int r = 0; r < D; ++r) {
            const int j = ((r - t) % D + D) % D;
            const bool last = t + 1 == D;
            // running state: straight into out / lse when they are fp32, else
            // in fp32 in the workspace until the last step writes out
            const bool in_place = out_dtype == ST_DTYPE_F32;
            float* st_out = in_place ? static_cast<float*>(out[r]) : run_out(r);
            float* st_lse = in_place ? lse[r] : run_lse(r);
            void* dst_out = last ? out[r] : st_out;
            float* dst_lse = last ? lse[r] : st_lse;
            const int dst_dtype = last ? out_dtype : ST_DTYPE_F32;
            rc = st_ring_fwd_step(L, r, j, B, H, d, ST_DTYPE_BF16, causal, scale, q[r], held_k(r, t), held_v(r, t),
                                  t == 0 ? nullptr : st_out, t == 0 ? nullptr : st_lse, dst_dtype, dst_out, dst_lse,
                                  step_ws, w.step, stream);
            if (rc != ST_OK) return rc;
        }
        if ((rc = ck(cudaEventRecord(e.ev[1 + t], cs))) != ST_OK) return rc;
    }
    // `stream` completes after every copy
    if ((rc = ck(cudaEventRecord(e.ev[0], xs))) != ST_OK) return rc;
    return ck(cudaStreamWaitEvent(cs, e.ev[0], 0));
}

extern "C" int st_ring_bwd_local(const st_layout_t* L, int B, int H, int d, int causal, float scale,
                                 const void* const* q, const void* const* k, const void* const* v,
                                 const void* const* out, int out_dtype, const float* const* lse,
                                 const void* const* dout, float* const* dq, float* const* dk, float* const* dv,
                                 void* workspace, size_t ws_bytes, void* stream, void* copy_stream) {
    int rc = check_local(L, B, H, d, &scale, workspace, ws_bytes, 1, stream, copy_stream);
    if (rc != ST_OK) return rc;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    const int D = L->D;
    if ((rc = check_ptr_array(D, q)) || (rc = check_ptr_array(D, k)) || (rc = check_ptr_array(D, v)) ||
        (rc = check_ptr_array(D, out)) || (rc = check_ptr_array(D, lse)) || (rc = check_ptr_array(D, dout)) ||
        (rc = check_ptr_array(D, dq)) || (rc = check_ptr_array(D, dk)) || (rc = check_ptr_array(D, dv)))
        return rc;
    if (!ptr_array_on_device(D, q) || !ptr_array_on_device(D, k) || !ptr_array_on_device(D, v) ||
        !ptr_array_on_device(D, out) || !ptr_array_on_device(D, lse) || !ptr_array_on_device(D, dout) ||
        !ptr_array_on_device(D, dq) || !ptr_array_on_device(D, dk) || !ptr_array_on_device(D, dv) ||
        !on_device(workspace))
        return ST_ERR_NOT_DEVICE;
    const LocalRing w = local_layout(*L, B, H, d, 1);
    char* ws = static_cast<char*>(workspace);
    // per rank and slot: K, V (bf16), dK, dV accumulators (fp32)
    auto slot_base = [&](int r, int s) { return ws + r * w.per_rank + s * (2 * w.blk16 + 2 * w.blk32); };
    auto buf_k = [&](int r, int s) { return slot_base(r, s); };
    auto buf_v = [&](int r, int s) { return slot_base(r, s) + w.blk16; };
    auto acc_k = [&](int r, int s) { return reinterpret_cast<float*>(slot_base(r, s) + 2 * w.blk16); };
    auto acc_v = [&](int r, int s) { return reinterpret_cast<float*>(slot_base(r, s) + 2 * w.blk16 + w.blk32); };
    void* step_ws = ws + (size_t)D * w.per_rank;
    cudaStream_t cs = static_cast<cudaStream_t>(stream), xs = static_cast<cudaStream_t>(copy_stream);
    Events e;
    // ev[0]: entry / exit; kv_sent[t] = ev[1 + t] (K/V of step t in slot t & 1);
    // computed[t] = ev[1 + D + t]; acc_sent[t] = ev[1 + 2D + t]
    if ((rc = e.make(1 + 3 * D)) != ST_OK) return rc;
    auto ck = [](cudaError_t x) { return cuda_status((int)x); };
    const size_t row16 = (size_t)H * d * 2, row32 = (size_t)H * d * 4;
    // every rank starts with its own K/V shard and zero dK/dV accumulators
    for (int r = 0; r < D; ++r) {
        const size_t n = (size_t)B * L->lens[r];
        if ((rc = ck(cudaMemsetAsync(acc_k(r, 0), 0, n * row32, cs))) != ST_OK) return rc;
        if ((rc = ck(cudaMemsetAsync(acc_v(r, 0), 0, n * row32, cs))) != ST_OK) return rc;
    }
    if ((rc = ck(cudaEventRecord(e.ev[0], cs))) != ST_OK) return rc;
    if ((rc = ck(cudaStreamWaitEvent(xs, e.ev[0], 0))) != ST_OK) return rc;
    auto held_k = [&](int r, int t) -> const void* { return t == 0 ? k[r] : buf_k(r, t & 1); };
    auto held_v = [&](int r, int t) -> const void* { return t == 0 ? v[r] : buf_v(r, t & 1); };
    for (int t = 0; t < D; ++t) {
        // K and V of step t + 1 travel while step t computes (read-only there);
        // the slot they overwrite was last used by step t - 1
        if (t + 1 < D) {
            if (t >= 1 && (rc = ck(cudaStreamWaitEvent(xs, e.ev[1 + D + t - 1], 0))) != ST_OK) return rc;
            for (int r = 0; r < D; ++r) {
                const int src = (r + D - 1) % D;
                const int j = ((src - t) % D + D) % D;
                const size_t n = (size_t)B * L->lens[j] * row16;
                if ((rc = ck(cudaMemcpyAsync(buf_k(r, (t + 1) & 1), held_k(src, t), n, cudaMemcpyDeviceToDevice,
                                             xs))) != ST_OK ||
                    (rc = ck(cudaMemcpyAsync(buf_v(r, (t + 1) & 1), held_v(src, t), n, cudaMemcpyDeviceToDevice,
                                             xs))) != ST_OK)
                    return rc;
            }
            if ((rc = ck(cudaEventRecord(e.ev[1 + t + 1], xs))) != ST_OK) return rc;
        }
        if (t >= 1) {
            if ((rc = ck(cudaStreamWaitEvent(cs, e.ev[1 + t], 0))) != ST_OK) return rc;
            if ((rc = ck(cudaStreamWaitEvent(cs, e.ev[1 + 2 * D + t], 0))) != ST_OK) return rc;
        }
        for (int r = 0; r < D; ++r) {
            const int j = ((r - t) % D + D) % D;
            rc = bwd_step(*L, r, j, B, H, d, causal ? 1 : 0, scale, q[r], held_k(r, t), held_v(r, t), out[r],
                          out_dtype, lse[r], dout[r], t == 0 ? 1 : 0, dq[r], acc_k(r, t & 1), acc_v(r, t & 1),
                          step_ws, stream);
            if (rc != ST_OK) return rc;
        }
        if ((rc = ck(cudaEventRecord(e.ev[1 + D + t], cs))) != ST_OK) return rc;
        // the accumulators move on once step t has added to them: to the next
        // rank for step t + 1, or after the last step home to the shard's owner
        if ((rc = ck(cudaStreamWaitEvent(xs, e.ev[1 + D + t], 0))) != ST_OK) return rc;
        for (int r = 0; r < D; ++r) {
            const int dst = (r + 1) % D;
            const int j = ((r - t) % D + D) % D;
            const size_t n = (size_t)B * L->lens[j] * row32;
            void* to_k = t + 1 < D ? static_cast<void*>(acc_k(dst, (t + 1) & 1)) : static_cast<void*>(dk[j]);
            void* to_v = t + 1 < D ? static_cast<void*>(acc_v(dst, (t + 1) & 1)) : static_cast<void*>(dv[j]);
            if ((rc = ck(cudaMemcpyAsync(to_k, acc_k(r, t & 1), n, cudaMemcpyDeviceToDevice, xs))) != ST_OK ||
                (rc = ck(cudaMemcpyAsync(to_v, acc_v(r, t & 1), n, cudaMemcpyDeviceToDevice, xs))) != ST_OK)
                return rc;
        }
        if (t + 1 < D && (rc = ck(cudaEventRecord(e.ev[1 + 2 * D + t + 1], xs))) != ST_OK) return rc;
    }
    if ((rc = ck(cudaEventRecord(e.ev[0], xs))) != ST_OK) return rc;
    return ck(cudaStreamWaitEvent(cs, e.ev[0], 0));
}
