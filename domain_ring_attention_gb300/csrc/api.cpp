// C-ABI entry points: argument validation and dispatch to the kernels.
// Every check happens on the host before anything is launched, so an invalid
// call returns an error code and never reaches the GPU.
#include <cmath>
#include <cstdint>

#include <cuda_runtime_api.h>

#include <algorithm>
#include <vector>

#include "common.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_status(int err) {
    if (err == 0) return ST_OK;
    g_last_cuda_error = err;
    return ST_ERR_CUDA;
}

using st::aligned16;
using st::on_device;

template <typename... P>
bool all_on_device(P... ps) {
    return (on_device(ps) && ...);
}

// The GEMM kernels count output tiles (128 x 128 at the finest) in int.
bool gemm_tiles_fit(int64_t M, int64_t N) { return ((M + 127) / 128) * ((N + 127) / 128) < ((int64_t)1 << 31); }

bool shards_on_device(int D, void* const* shards) {
    for (int r = 0; r < D; ++r)
        if (!on_device(shards[r])) return false;
    return true;
}

int check_common(const st_layout_t* L, int B, int H, int d, int dtype, float* scale) {
    if (!L) return ST_ERR_NULL;
    if (B < 1 || H < 1 || (int64_t)B * H > 65535) return ST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ST_ERR_UNSUPPORTED;
    if (dtype != ST_DTYPE_F32 && dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!std::isfinite(*scale)) return ST_ERR_INVALID_ARG;
    if (*scale <= 0.f) *scale = 1.0f / std::sqrt((float)d);
    return ST_OK;
}

}  // namespace

extern "C" const char* st_error_string(int code) {
    switch (code) {
        case ST_OK: return "ok";
        case ST_ERR_NULL: return "a required pointer is NULL";
        case ST_ERR_INVALID_LAYOUT: return "invalid sharding shapes (D, a length < 1, or an odd zigzag length)";
        case ST_ERR_UNSUPPORTED: return "unsupported head_dim or dtype";
        case ST_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned";
        case ST_ERR_WORKSPACE: return "workspace missing or too small";
        case ST_ERR_CUDA: return "CUDA error (see st_last_cuda_error)";
        case ST_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
        case ST_ERR_INVALID_ARG: return "an argument is out of range";
        case ST_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed 32 MiB scratch of st_attn_fwd_noalloc";
        case ST_ERR_NOT_DEVICE: return "a pointer that must address device memory does not";
        default: return "unknown status";
    }
}

extern "C" int st_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int st_is_device_pointer(const void* p) { return p && on_device(p) ? 1 : 0; }

extern "C" int st_device_error(void* stream) {
    int rc = cuda_status((int)cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    if (rc != ST_OK) return rc;
    const int f = st::fwd_tc_device_error(true);
    const int b = st::bwd_tc_device_error(true);
    const int g = st::gemm_tc_device_error(true);
    const int c = st::conv_tc_device_error(true);
    const int t = st::selftest_device_error(true);
    if (f < 0 || b < 0 || g < 0 || c < 0 || t < 0) return cuda_status((int)cudaGetLastError());
    return (f || b || g || c || t) ? ST_ERR_DEVICE_TIMEOUT : ST_OK;
}

extern "C" int st_proj_gemm(int M, int N, int K, const void* x, const void* w, void* y, int out_dtype,
                            void* stream) {
    if (!x || !w || !y) return ST_ERR_NULL;
    if (M < 1 || N < 1 || K < 1 || N % 8 != 0 || K % 8 != 0 || !gemm_tiles_fit(M, N)) return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_BF16 && out_dtype != ST_DTYPE_F32) return ST_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return ST_ERR_MISALIGNED;
    if (!all_on_device(x, w, y)) return ST_ERR_NOT_DEVICE;
    return cuda_status(st::launch_gemm_tc(M, N, K, x, w, y, out_dtype, stream));
}

namespace {

// shared checks of the sharded-image entry points; rows are host values
int check_image_shards(int D, const int64_t* rows, int W, void* const* shards) {
    if (!rows || !shards) return ST_ERR_NULL;
    if (D < 1 || D > ST_CONV_MAX_SHARDS || W < 1) return ST_ERR_INVALID_ARG;
    int64_t H = 0;
    for (int r = 0; r < D; ++r) {
        if (rows[r] < 1) return ST_ERR_INVALID_LAYOUT;
        H += rows[r];
        if (!shards[r]) return ST_ERR_NULL;
        if (!aligned16(shards[r])) return ST_ERR_MISALIGNED;
    }
    if (H > (1 << 24)) return ST_ERR_INVALID_ARG;
    return ST_OK;
}

}  // namespace

extern "C" int st_halo_exchange(int D, const int64_t* rows, int W, int C, int halo, void* const* shards,
                                void* stream) {
    int rc = check_image_shards(D, rows, W, shards);
    if (rc != ST_OK) return rc;
    if (C < 8 || C % 8 != 0 || halo < 0 || halo > 3) return ST_ERR_INVALID_ARG;
    if ((int64_t)W * C > (1 << 24)) return ST_ERR_INVALID_ARG;
    if (!shards_on_device(D, shards)) return ST_ERR_NOT_DEVICE;
    return cuda_status(st::launch_halo_exchange(D, rows, W, C, halo, shards, stream));
}

extern "C" int st_conv2d_sharded(int D, const int64_t* rows, int W, int C_in, int C_out, int k,
                                 void* const* in_shards, const void* weight, const float* bias,
                                 void* const* out_shards, int out_dtype, void* stream) {
    int rc = check_image_shards(D, rows, W, in_shards);
    if (rc != ST_OK) return rc;
    rc = check_image_shards(D, rows, W, out_shards);
    if (rc != ST_OK) return rc;
    if (!weight) return ST_ERR_NULL;
    if (k < 1 || k > 7 || k % 2 == 0 || C_in < 64 || C_in % 64 != 0 || C_in > 4096 || C_out < 8 ||
        C_out % 8 != 0 || C_out > 4096)
        return ST_ERR_INVALID_ARG;
    int64_t H = 0;
    for (int r = 0; r < D; ++r) H += rows[r];
    // the kernel counts (row, 128-pixel tile, channel tile) units in int
    if (H * ((W + 127) / 128) * ((C_out + 127) / 128) >= ((int64_t)1 << 31)) return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_BF16 && out_dtype != ST_DTYPE_F32) return ST_ERR_UNSUPPORTED;
    if (!aligned16(weight) || (bias && reinterpret_cast<uintptr_t>(bias) % 4 != 0)) return ST_ERR_MISALIGNED;
    if (!shards_on_device(D, in_shards) || !shards_on_device(D, out_shards) || !all_on_device(weight, bias))
        return ST_ERR_NOT_DEVICE;
    return cuda_status(
        st::launch_conv_tc(D, rows, W, C_in, C_out, k, in_shards, weight, bias, out_shards, out_dtype, stream));
}

namespace {

int check_group_norm(int C, int G) {
    // C / 8 vectors per pixel must divide the 256 threads of a block
    if (C < 8 || C > 2048 || (C & (C - 1)) != 0) return ST_ERR_INVALID_ARG;
    if (G < 1 || C % G != 0 || (C / G) % 8 != 0) return ST_ERR_INVALID_ARG;
    return ST_OK;
}

}  // namespace

extern "C" int st_group_norm_workspace_size(int C, int G, size_t* bytes) {
    if (!bytes) return ST_ERR_NULL;
    const int rc = check_group_norm(C, G);
    if (rc != ST_OK) return rc;
    *bytes = st::group_norm_workspace_bytes(G);
    return ST_OK;
}

extern "C" int st_group_norm_sharded(int D, const int64_t* rows, int W, int C, int G, float eps,
                                     const void* const* in_shards, const float* gamma, const float* beta,
                                     void* const* out_shards, int out_pad, int out_dtype, void* workspace,
                                     size_t ws_bytes, void* stream) {
    int rc = check_image_shards(D, rows, W, const_cast<void* const*>(in_shards));
    if (rc != ST_OK) return rc;
    rc = check_image_shards(D, rows, W, out_shards);
    if (rc != ST_OK) return rc;
    rc = check_group_norm(C, G);
    if (rc != ST_OK) return rc;
    if (!(eps > 0.f) || out_pad < 0 || out_pad > 3) return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_BF16 && out_dtype != ST_DTYPE_F32) return ST_ERR_UNSUPPORTED;
    if ((gamma && reinterpret_cast<uintptr_t>(gamma) % 4) || (beta && reinterpret_cast<uintptr_t>(beta) % 4))
        return ST_ERR_MISALIGNED;
    if (!workspace) return ST_ERR_WORKSPACE;
    if (ws_bytes < st::group_norm_workspace_bytes(G)) return ST_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
    if (!shards_on_device(D, const_cast<void* const*>(in_shards)) || !shards_on_device(D, out_shards) ||
        !all_on_device(gamma, beta, workspace))
        return ST_ERR_NOT_DEVICE;
    return cuda_status(st::launch_group_norm(D, rows, W, C, G, eps, in_shards, gamma, beta, out_shards, out_pad,
                                             out_dtype, workspace, stream));
}

extern "C" int st_gated_mlp(int M, int hidden, int F, const void* x, const void* w1, const void* w3,
                            const void* w2, void* h, void* y, int out_dtype, void* stream) {
    if (!x || !w1 || !w3 || !w2 || !h || !y) return ST_ERR_NULL;
    if (M < 1 || hidden < 1 || F < 1 || hidden % 8 != 0 || F % 8 != 0 || !gemm_tiles_fit(M, F) ||
        !gemm_tiles_fit(M, hidden))
        return ST_ERR_INVALID_ARG;
    if (out_dtype != ST_DTYPE_BF16 && out_dtype != ST_DTYPE_F32) return ST_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) || !aligned16(h) || !aligned16(y))
        return ST_ERR_MISALIGNED;
    if (!all_on_device(x, w1, w3, w2, h, y)) return ST_ERR_NOT_DEVICE;
    int rc = cuda_status(st::launch_gemm_gated(M, F, hidden, x, w1, w3, h, stream));
    if (rc != ST_OK) return rc;
    return cuda_status(st::launch_gemm_tc(M, hidden, F, h, w2, y, out_dtype, stream));
}

namespace st {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Memory the kernels may read and write: device or managed allocations.  A
// pointer to ordinary host memory handed to a kernel would fault the GPU, so
// every entry point checks its device pointers with the runtime, after all its
// other checks (so argument errors are still reported without a GPU).  NULL
// is accepted here (optional arguments were checked before).
bool on_device(const void* p) {
    if (!p) return true;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // do not leave the failure to be read as a launch error
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

BwdWorkspace bwd_workspace_layout(int64_t rows, int d, int dtype) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    BwdWorkspace w;
    size_t off = 0;
    w.dq_acc = off;
    off += up((size_t)rows * d * sizeof(float));
    w.delta = off;
    off += up((size_t)rows * sizeof(float));
    w.stats = off;
    if (dtype == ST_DTYPE_F32) off += up(2 * (size_t)rows * sizeof(double));
    w.h16 = off;
    if (dtype == ST_DTYPE_BF16) off += 4 * up((size_t)rows * d * 2);
    w.scales = off;
    off += 256;
    w.total = off;
    return w;
}

int record_cuda_error(int err) { return cuda_status(err); }

size_t fwd_workspace_bytes(int64_t rows, int d, int dtype) {
    if (dtype != ST_DTYPE_BF16) return 0;
    return (((size_t)rows * d * 2 + 255) & ~(size_t)255) + 256;
}

}  // namespace st

extern "C" int st_attn_workspace_size(const st_layout_t* L, int B, int H, int d, int dtype,
                                      int pass, size_t* bytes) {
    float scale = 1.f;
    if (!bytes) return ST_ERR_NULL;
    const int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (pass == 0) {
        *bytes = st::fwd_workspace_bytes((int64_t)B * L->S * H, d, dtype);
    } else if (pass == 1) {
        *bytes = st::bwd_workspace_layout((int64_t)B * L->S * H, d, dtype).total;
    } else {
        return ST_ERR_INVALID_ARG;
    }
    return ST_OK;
}

extern "C" int st_attn_fwd(const st_layout_t* L, int B, int H, int d, int dtype, int causal,
                           float scale, const void* q, const void* k, const void* v, int out_dtype,
                           void* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != dtype) return ST_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || !lse) return ST_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return ST_ERR_MISALIGNED;
    st::AttnArgs a{q, k, v, out, lse, nullptr, nullptr, B, H, d, causal ? 1 : 0, scale, out_dtype,
                   nullptr, nullptr, nullptr};
    if (dtype == ST_DTYPE_BF16) {
        const int64_t rows = (int64_t)B * L->S * H;
        const size_t need = st::fwd_workspace_bytes(rows, d, dtype);
        if (!workspace || ws_bytes < need) return ST_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
        if (!all_on_device(q, k, v, out, lse, workspace)) return ST_ERR_NOT_DEVICE;
        char* ws = static_cast<char*>(workspace);
        a.v16 = ws;
        a.amax_bits = reinterpret_cast<unsigned*>(ws + need - 256);
        a.exps = reinterpret_cast<int*>(ws + need - 128);
        rc = cuda_status(st::launch_fp16_copy1(v, a.v16, rows * d, a.amax_bits, a.exps, stream));
        if (rc != ST_OK) return rc;
        bool handled = false;
        rc = st::launch_fwd_tc(*L, a, stream, &handled);
        if (handled) return cuda_status(rc);
        return ST_ERR_UNSUPPORTED;
    }
    if (!all_on_device(q, k, v, out, lse)) return ST_ERR_NOT_DEVICE;
    st::SegTable t;
    st::fill_segtable(*L, 64, &t);
    return cuda_status(st::launch_fwd_simt(t, a, dtype, stream));
}

namespace {

// st_attn_fwd_host with the heads in groups: per group, the 2-D copies of its
// heads' V, K and Q (pitch H * d), the exact fp16 copy of its V with an
// exponent of its own, the attention launch over its heads, and its output
// and lse copied back.  Groups alternate between `stream` and a second stream
// made here, so that one group's last wave overlaps the next group's first.
int fwd_host_groups(const st_layout_t* L, const st::SegTable& t, int B, int H, int d, int causal, float scale,
                    int hn_mid, const void* q_host, const void* k_host, const void* v_host, void* out_host,
                    float* lse_host, void* q, void* k, void* v, void* out, float* lse, void* workspace,
                    size_t need, void* stream, void* copy_stream) {
    // group boundaries: a single head first and last (little to copy in before
    // the first launch, little to copy back after the last), hn_mid between
    std::vector<int> hb{0};
    if (H >= 3) hb.push_back(1);
    while (hb.back() < H - 1) hb.push_back(std::min(H - 1, hb.back() + hn_mid));
    if (hb.back() < H) hb.push_back(H);
    const int G = (int)hb.size() - 1;
    const int64_t S = L->S;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
    cudaStream_t s2 = nullptr;
    // ev[0]: work queued on `stream` before this call, later the last copy
    // back; per group g: V landed (1 + 3g), K and Q landed (2 + 3g), computed (3 + 3g)
    std::vector<cudaEvent_t> ev(1 + 3 * G, nullptr);
    int rc = ST_OK;
    auto ck = [&](cudaError_t e) { return cuda_status((int)e); };
    auto finish = [&](int code) {
        for (auto& e : ev)
            if (e) cudaEventDestroy(e);   // released once pending work has passed it
        if (s2) cudaStreamDestroy(s2);    // likewise: its queued work still runs
        return code;
    };
    for (auto& e : ev)
        if ((rc = ck(cudaEventCreateWithFlags(&e, cudaEventDisableTiming))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking))) != ST_OK) return finish(rc);
    const size_t pitch = (size_t)H * d * 2;        // one token of q, k, v or out (bf16)
    const size_t hw = (size_t)d * 2;               // one head within it
    const size_t rows = (size_t)B * S;
    // everything queued on `stream` before this call comes first on all three streams
    if ((rc = ck(cudaEventRecord(ev[0], cs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamWaitEvent(xs, ev[0], 0))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamWaitEvent(s2, ev[0], 0))) != ST_OK) return finish(rc);
    for (int g = 0; g < G; ++g) {
        const size_t off = (size_t)hb[g] * hw, gw = (size_t)(hb[g + 1] - hb[g]) * hw;
        auto h2d = [&](void* dst, const void* src) {
            return ck(cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, static_cast<const char*>(src) + off,
                                        pitch, gw, rows, cudaMemcpyHostToDevice, xs));
        };
        if ((rc = h2d(v, v_host)) != ST_OK) return finish(rc);
        if ((rc = ck(cudaEventRecord(ev[1 + 3 * g], xs))) != ST_OK) return finish(rc);
        if ((rc = h2d(k, k_host)) != ST_OK) return finish(rc);
        if ((rc = h2d(q, q_host)) != ST_OK) return finish(rc);
        if ((rc = ck(cudaEventRecord(ev[2 + 3 * g], xs))) != ST_OK) return finish(rc);
    }
    char* ws = static_cast<char*>(workspace);
    unsigned* amax = reinterpret_cast<unsigned*>(ws + need - 256);   // one per group (G <= 18 < 32)
    int* exps = reinterpret_cast<int*>(ws + need - 128);
    for (int g = 0; g < G; ++g) {
        cudaStream_t gs = (g & 1) ? s2 : cs;
        const int hn = hb[g + 1] - hb[g];
        const size_t off = (size_t)hb[g] * hw, gw = (size_t)hn * hw;
        if ((rc = ck(cudaStreamWaitEvent(gs, ev[1 + 3 * g], 0))) != ST_OK) return finish(rc);
        // the fp16 copy of V lives at the same offsets as V (2 bytes per element)
        if ((rc = cuda_status(st::launch_fp16_copy_rows(static_cast<char*>(v) + off, ws + off, (int64_t)rows,
                                                        (int)(gw / 16), (int64_t)(pitch / 16), amax + g, exps + g,
                                                        gs))) != ST_OK)
            return finish(rc);
        if ((rc = ck(cudaStreamWaitEvent(gs, ev[2 + 3 * g], 0))) != ST_OK) return finish(rc);
        st::AttnArgs a{q, k, v, out, lse, nullptr, nullptr, B, H, d, causal ? 1 : 0, scale, ST_DTYPE_BF16,
                       ws, amax + g, exps + g};
        a.h0 = hb[g];
        a.hn = hn;
        bool handled = false;
        rc = st::launch_fwd_tc(*L, a, gs, &handled, 0, t.ntiles);
        if (!handled) return finish(ST_ERR_UNSUPPORTED);
        if ((rc = cuda_status(rc)) != ST_OK) return finish(rc);
        if ((rc = ck(cudaEventRecord(ev[3 + 3 * g], gs))) != ST_OK) return finish(rc);
        // this group's output and lse back to the host while the next group runs
        if ((rc = ck(cudaStreamWaitEvent(xs, ev[3 + 3 * g], 0))) != ST_OK) return finish(rc);
        if ((rc = ck(cudaMemcpy2DAsync(static_cast<char*>(out_host) + off, pitch, static_cast<const char*>(out) + off,
                                       pitch, gw, rows, cudaMemcpyDeviceToHost, xs))) != ST_OK)
            return finish(rc);
        // lse [B, H, S]: the group's hn * S values of every batch entry
        const size_t lo = (size_t)hb[g] * S;
        if ((rc = ck(cudaMemcpy2DAsync(lse_host + lo, (size_t)H * S * 4, lse + lo, (size_t)H * S * 4,
                                       (size_t)hn * S * 4, (size_t)B, cudaMemcpyDeviceToHost, xs))) != ST_OK)
            return finish(rc);
    }
    // `stream` completes only after the last copy back (which follows every group)
    if ((rc = ck(cudaEventRecord(ev[0], xs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamWaitEvent(cs, ev[0], 0))) != ST_OK) return finish(rc);
    return finish(ST_OK);
}

}  // namespace

extern "C" int st_attn_fwd_host(const st_layout_t* L, int B, int H, int d, int dtype, int causal, float scale,
                                const void* q_host, const void* k_host, const void* v_host, void* out_host,
                                float* lse_host, void* q, void* k, void* v, void* out, float* lse,
                                void* workspace, size_t ws_bytes, void* stream, void* copy_stream) {
    int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!q_host || !k_host || !v_host || !out_host || !lse_host || !q || !k || !v || !out || !lse)
        return ST_ERR_NULL;
    if (!copy_stream || copy_stream == stream) return ST_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return ST_ERR_MISALIGNED;
    const int64_t S = L->S;
    const int64_t rows = (int64_t)B * S * H;
    const size_t need = st::fwd_workspace_bytes(rows, d, dtype);
    if (!workspace || ws_bytes < need) return ST_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
    if (!all_on_device(q, k, v, out, lse, workspace)) return ST_ERR_NOT_DEVICE;

    // Query tiles (256 rows of one segment each, in buffer order) and the
    // buffer rows they start at.
    st::SegTable t;
    const int tile_rows = st::fwd_tc_tile_rows();
    st::fill_segtable(*L, tile_rows, &t);
    auto tile_row = [&](int tl) -> int64_t {   // first buffer row of tile tl (tl == ntiles: S)
        if (tl >= t.ntiles) return S;
        int sgm = 0;
        while (t.seg_tile[sgm + 1] <= tl) ++sgm;
        return t.seg_buf[sgm] + (int64_t)(tl - t.seg_tile[sgm]) * tile_rows;
    };
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // Heads in groups, when groups of hn heads still make launches of at least
    // four waves of CTAs (a single head first and last, hn between): every query
    // tile needs all of its head's K and V, so with groups only the first
    // group's K, V (and Q) stand before the first launch, the rest arriving
    // while earlier groups compute, and only the last group's output is copied
    // back after the compute.
    int hn = H;
    for (int g = 2; g <= std::min(H, 16); ++g) {
        if (H % g) continue;
        if ((int64_t)t.ntiles * B * (H / g) < 4LL * std::max(sms, 1)) break;
        hn = H / g;
    }
    // H without such a divisor (a prime, say): the fewest heads that make four
    // waves, and at least (H - 2) / 16 (at most 18 groups: the workspace holds
    // 32 exponents), when the whole problem spans eight waves or more
    const int64_t per_head = (int64_t)t.ntiles * B;
    if (hn == H && H >= 4 && per_head * H >= 8LL * std::max(sms, 1)) {
        int want = (int)((4LL * std::max(sms, 1) + per_head - 1) / per_head);
        want = std::max(want, (H - 2 + 15) / 16);
        if (want <= H - 2) hn = want;
    }
    if (hn < H)
        return fwd_host_groups(L, t, B, H, d, causal, scale, hn, q_host, k_host, v_host, out_host, lse_host, q, k,
                               v, out, lse, workspace, need, stream, copy_stream);
    // Chunks of query tiles: a short first chunk (about two waves of CTAs) so
    // that compute starts early while the rest of Q arrives, a short last
    // chunk so that little output is left to copy back after compute ends, and
    // the bulk in between (whole waves where possible).
    const int per_tile = B * H;                          // CTAs per query tile
    const int edge = std::max(1, (2 * std::max(sms, 1) + per_tile - 1) / per_tile);
    std::vector<int> cuts{0};
    if (t.ntiles > 4 * edge) {
        cuts.push_back(edge);
        cuts.push_back(t.ntiles - edge);
    }
    cuts.push_back(t.ntiles);
    const int nchunks = (int)cuts.size() - 1;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaStream_t xs = static_cast<cudaStream_t>(copy_stream);
    // ev[0]: work queued on `stream` before this call, then V landed, then the
    // last copy back; ev[1 .. nchunks]: Q chunk c landed; the rest: chunk c computed
    std::vector<cudaEvent_t> ev(1 + 2 * nchunks, nullptr);
    for (auto& e : ev)
        if ((rc = cuda_status((int)cudaEventCreateWithFlags(&e, cudaEventDisableTiming))) != ST_OK) break;
    auto finish = [&](int code) {
        for (auto& e : ev)
            if (e) cudaEventDestroy(e);   // released once pending work has passed it
        return code;
    };
    if (rc != ST_OK) return finish(rc);
    const size_t row_bytes = (size_t)H * d * 2;            // one token of q, k, v or out (bf16)
    const size_t kv_bytes = (size_t)B * S * row_bytes;
    auto ck = [&](cudaError_t e) { return cuda_status((int)e); };
    // The copies into q, k, v (and out of out, lse) must come after everything
    // already queued on `stream`, which may still read or write those buffers
    // (or memory that a stream-ordered allocator has just handed them).
    if ((rc = ck(cudaEventRecord(ev[0], cs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamWaitEvent(xs, ev[0], 0))) != ST_OK) return finish(rc);
    // V, then K: every query tile needs all of both; the fp16 copy of V runs
    // while K is still coming in
    if ((rc = ck(cudaMemcpyAsync(v, v_host, kv_bytes, cudaMemcpyHostToDevice, xs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaEventRecord(ev[0], xs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaMemcpyAsync(k, k_host, kv_bytes, cudaMemcpyHostToDevice, xs))) != ST_OK) return finish(rc);
    for (int c = 0; c < nchunks; ++c) {
        const int64_t r0 = tile_row(cuts[c]), r1 = tile_row(cuts[c + 1]);
        for (int b = 0; b < B; ++b) {
            const size_t off = ((size_t)b * S + r0) * row_bytes;
            if ((rc = ck(cudaMemcpyAsync(static_cast<char*>(q) + off, static_cast<const char*>(q_host) + off,
                                         (size_t)(r1 - r0) * row_bytes, cudaMemcpyHostToDevice, xs))) != ST_OK)
                return finish(rc);
        }
        if ((rc = ck(cudaEventRecord(ev[1 + c], xs))) != ST_OK) return finish(rc);
    }
    // compute: the fp16 copy of V once V is in, then each chunk once its Q rows
    // are in (they follow K on the copy stream)
    st::AttnArgs a{q, k, v, out, lse, nullptr, nullptr, B, H, d, causal ? 1 : 0, scale, ST_DTYPE_BF16,
                   nullptr, nullptr, nullptr};
    char* ws = static_cast<char*>(workspace);
    a.v16 = ws;
    a.amax_bits = reinterpret_cast<unsigned*>(ws + need - 256);
    a.exps = reinterpret_cast<int*>(ws + need - 128);
    if ((rc = ck(cudaStreamWaitEvent(cs, ev[0], 0))) != ST_OK) return finish(rc);
    if ((rc = cuda_status(st::launch_fp16_copy1(v, a.v16, rows * d, a.amax_bits, a.exps, stream))) != ST_OK)
        return finish(rc);
    for (int c = 0; c < nchunks; ++c) {
        if ((rc = ck(cudaStreamWaitEvent(cs, ev[1 + c], 0))) != ST_OK) return finish(rc);
        bool handled = false;
        rc = st::launch_fwd_tc(*L, a, stream, &handled, cuts[c], cuts[c + 1]);
        if (!handled) return finish(ST_ERR_UNSUPPORTED);
        if ((rc = cuda_status(rc)) != ST_OK) return finish(rc);
        if ((rc = ck(cudaEventRecord(ev[1 + nchunks + c], cs))) != ST_OK) return finish(rc);
        // that chunk's output rows and lse back to the host while the next chunk runs
        if ((rc = ck(cudaStreamWaitEvent(xs, ev[1 + nchunks + c], 0))) != ST_OK) return finish(rc);
        const int64_t r0 = tile_row(cuts[c]), r1 = tile_row(cuts[c + 1]);
        for (int b = 0; b < B; ++b) {
            const size_t off = ((size_t)b * S + r0) * row_bytes;
            if ((rc = ck(cudaMemcpyAsync(static_cast<char*>(out_host) + off, static_cast<const char*>(out) + off,
                                         (size_t)(r1 - r0) * row_bytes, cudaMemcpyDeviceToHost, xs))) != ST_OK)
                return finish(rc);
        }
        // lse [B, H, S]: rows r0 .. r1 of every (b, h)
        if ((rc = ck(cudaMemcpy2DAsync(lse_host + r0, (size_t)S * 4, lse + r0, (size_t)S * 4, (size_t)(r1 - r0) * 4,
                                       (size_t)B * H, cudaMemcpyDeviceToHost, xs))) != ST_OK)
            return finish(rc);
    }
    // `stream` completes only after the last copy back
    if ((rc = ck(cudaEventRecord(ev[0], xs))) != ST_OK) return finish(rc);
    if ((rc = ck(cudaStreamWaitEvent(cs, ev[0], 0))) != ST_OK) return finish(rc);
    return finish(ST_OK);
}

extern "C" int st_attn_fwd_partials(const st_layout_t* L, int B, int H, int d, int dtype,
                                    int causal, float scale, const void* q, const void* k,
                                    const void* v, float* partial_out, float* partial_lse,
                                    void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (!q || !k || !v || !partial_out || !partial_lse) return ST_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(partial_out) ||
        !aligned16(partial_lse))
        return ST_ERR_MISALIGNED;
    st::AttnArgs a{q, k, v, nullptr, nullptr, partial_out, partial_lse, B, H, d, causal ? 1 : 0, scale,
                   ST_DTYPE_F32, nullptr, nullptr, nullptr};
    if (dtype == ST_DTYPE_BF16) {
        const int64_t rows = (int64_t)B * L->S * H;
        const size_t need = st::fwd_workspace_bytes(rows, d, dtype);
        if (!workspace || ws_bytes < need) return ST_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
        if (!all_on_device(q, k, v, partial_out, partial_lse, workspace)) return ST_ERR_NOT_DEVICE;
        // the tensor-core forward with its state written out (and restarted) per KV shard
        char* ws = static_cast<char*>(workspace);
        a.v16 = ws;
        a.amax_bits = reinterpret_cast<unsigned*>(ws + need - 256);
        a.exps = reinterpret_cast<int*>(ws + need - 128);
        rc = cuda_status(st::launch_fp16_copy1(v, a.v16, rows * d, a.amax_bits, a.exps, stream));
        if (rc != ST_OK) return rc;
        bool handled = false;
        rc = st::launch_fwd_tc(*L, a, stream, &handled);
        if (handled) return cuda_status(rc);
        return ST_ERR_UNSUPPORTED;
    }
    if (!all_on_device(q, k, v, partial_out, partial_lse)) return ST_ERR_NOT_DEVICE;
    st::SegTable t;
    st::fill_segtable(*L, 64, &t);
    return cuda_status(st::launch_fwd_simt(t, a, dtype, stream));
}

extern "C" int st_attn_merge(int D, int B, int H, int64_t S, int d, const float* partial_out,
                             const float* partial_lse, void* out, float* lse, int out_dtype,
                             void* stream) {
    if (!partial_out || !partial_lse || !out || !lse) return ST_ERR_NULL;
    if (D < 1 || D > ST_MAX_SHARDS || B < 1 || H < 1 || S < 1 || S >= INT32_MAX)
        return ST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ST_ERR_UNSUPPORTED;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!aligned16(partial_out) || !aligned16(partial_lse) || !aligned16(out) || !aligned16(lse))
        return ST_ERR_MISALIGNED;
    if (!all_on_device(partial_out, partial_lse, out, lse)) return ST_ERR_NOT_DEVICE;
    return cuda_status(st::launch_merge(D, B, H, S, d, partial_out, partial_lse, out, lse,
                                        out_dtype, stream));
}

extern "C" int st_attn_bwd(const st_layout_t* L, int B, int H, int d, int dtype, int causal,
                           float scale, const void* q, const void* k, const void* v,
                           const void* out, int out_dtype, const float* lse, const void* dout,
                           int grad_dtype, void* dq, void* dk, void* dv, void* workspace,
                           size_t ws_bytes, void* stream) {
    int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (grad_dtype != ST_DTYPE_F32 && grad_dtype != dtype) return ST_ERR_UNSUPPORTED;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != dtype) return ST_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return ST_ERR_NULL;
    const void* ptrs[] = {q, k, v, out, lse, dout, dq, dk, dv};
    for (const void* p : ptrs)
        if (!aligned16(p)) return ST_ERR_MISALIGNED;
    const int64_t rows = (int64_t)B * L->S * H;
    const st::BwdWorkspace w = st::bwd_workspace_layout(rows, d, dtype);
    if (!workspace || ws_bytes < w.total) return ST_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ST_ERR_MISALIGNED;
    if (!all_on_device(q, k, v, out, lse, dout, dq, dk, dv, workspace)) return ST_ERR_NOT_DEVICE;
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
    // fp32 gradients accumulate straight into dq; otherwise into the workspace
    a.dq_acc = grad_dtype == ST_DTYPE_F32 ? static_cast<float*>(dq) : reinterpret_cast<float*>(ws + w.dq_acc);
    a.delta = reinterpret_cast<float*>(ws + w.delta);
    a.B = B;
    a.H = H;
    a.d = d;
    a.causal = causal ? 1 : 0;
    a.scale = scale;
    a.grad_dtype = grad_dtype;
    a.out_dtype = out_dtype;
    a.lse_d = reinterpret_cast<double*>(ws + w.stats);
    a.delta_d = a.lse_d + rows;
    const size_t plane = ((size_t)rows * d * 2 + 255) & ~(size_t)255;
    for (int i = 0; i < 4; ++i) a.h16[i] = ws + w.h16 + i * plane;
    a.amax_bits = reinterpret_cast<unsigned*>(ws + w.scales);
    a.exps = reinterpret_cast<int*>(ws + w.scales + 64);
    cudaStream_t st_ = static_cast<cudaStream_t>(stream);

    rc = cuda_status((int)cudaMemsetAsync(a.dq_acc, 0, (size_t)rows * d * sizeof(float), st_));
    if (rc != ST_OK) return rc;
    if (dtype == ST_DTYPE_F32) {
        st::SegTable t;
        st::fill_segtable(*L, 64, &t);
        rc = cuda_status(st::launch_rowstats_f64(t, a, stream));
        if (rc != ST_OK) return rc;
        rc = cuda_status(st::launch_bwd_simt(t, a, dtype, stream));
        if (rc != ST_OK) return rc;
    } else {
        rc = cuda_status(st::launch_bwd_preprocess(a, L->S, dtype, stream));
        if (rc != ST_OK) return rc;
        rc = cuda_status((int)cudaMemsetAsync(a.amax_bits, 0, 64, st_));
        if (rc != ST_OK) return rc;
        rc = cuda_status(st::launch_fp16_copies(a, L->S, stream));
        if (rc != ST_OK) return rc;
        bool handled = false;
        rc = cuda_status(st::launch_bwd_tc(*L, a, stream, &handled));
        if (rc != ST_OK) return rc;
        if (!handled) return ST_ERR_UNSUPPORTED;
    }
    if (grad_dtype == ST_DTYPE_F32) return ST_OK;
    return cuda_status(st::launch_dq_convert(a, L->S, grad_dtype, stream));
}

extern "C" int st_permute(const st_layout_t* L, int B, int H, int d, int dtype, int to_natural,
                          const void* in, void* out, void* stream) {
    float scale = 1.f;
    int rc = check_common(L, B, H, d, dtype, &scale);
    if (rc != ST_OK) return rc;
    if (!in || !out) return ST_ERR_NULL;
    if (in == out) return ST_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(out)) return ST_ERR_MISALIGNED;
    if (!all_on_device(in, out)) return ST_ERR_NOT_DEVICE;
    st::SegTable t;
    st::fill_segtable(*L, 64, &t);
    return cuda_status(st::launch_permute(t, B, H, d, dtype, to_natural ? 1 : 0, in, out, stream));
}

extern "C" int st_attn_bwd_delta(int B, int H, int64_t S, int d, int dtype, const void* out, int out_dtype,
                                 const void* dout, float* delta, void* stream) {
    if (!out || !dout || !delta) return ST_ERR_NULL;
    if (B < 1 || H < 1 || S < 1 || S >= INT32_MAX) return ST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ST_ERR_UNSUPPORTED;
    if (dtype != ST_DTYPE_F32 && dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (out_dtype != ST_DTYPE_F32 && out_dtype != dtype) return ST_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(dout) || !aligned16(delta)) return ST_ERR_MISALIGNED;
    if (!all_on_device(out, dout, delta)) return ST_ERR_NOT_DEVICE;
    st::BwdArgs a{};
    a.out = out;
    a.dout = dout;
    a.delta = delta;
    a.B = B;
    a.H = H;
    a.d = d;
    a.out_dtype = out_dtype;
    return cuda_status(st::launch_bwd_preprocess(a, S, dtype, stream));
}

extern "C" int st_convert_f32(int64_t n, const float* src, void* dst, int dst_dtype, void* stream) {
    if (!src || !dst) return ST_ERR_NULL;
    if (n < 1) return ST_ERR_INVALID_ARG;
    if (dst_dtype != ST_DTYPE_F32 && dst_dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    if (!aligned16(src) || !aligned16(dst)) return ST_ERR_MISALIGNED;
    if (!all_on_device(src, dst)) return ST_ERR_NOT_DEVICE;
    st::BwdArgs a{};
    a.dq_acc = const_cast<float*>(src);
    a.dq = dst;
    a.B = 1;
    a.H = 1;
    a.d = 1;
    return cuda_status(st::launch_dq_convert(a, n, dst_dtype, stream));
}

extern "C" int st_fp16_scaled_copy(int64_t n, const void* src, void* dst, int* exps, void* scratch, void* stream) {
    if (!src || !dst || !exps || !scratch) return ST_ERR_NULL;
    if (n < 8 || n % 8 != 0) return ST_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst) || !aligned16(exps) || !aligned16(scratch)) return ST_ERR_MISALIGNED;
    if (!all_on_device(src, dst, exps, scratch)) return ST_ERR_NOT_DEVICE;
    return cuda_status(st::launch_fp16_copy1(src, dst, n, static_cast<unsigned*>(scratch), exps, stream));
}
