// st_attn_fwd_noalloc: the forward for callers that cannot allocate device
// memory at all.
//
// st_attn_fwd needs a caller-provided workspace for bf16 inputs (the exact
// fp16 copy of v that feeds the P V product).  Some callers cannot provide
// one: code running inside another runtime's operator or plugin interface
// that hands it only its input and output buffers, real-time or safety-
// critical loops whose memory is fixed up front and forbid any allocation
// after start-up, and host code that must not touch a device allocator (whose
// calls synchronise and can fail for lack of memory) on its critical path.
// For them the scratch lives in a file-scope device array that is part of
// the loaded module: every GPU that loads the library holds it (32 MiB) until
// the process exits, and nothing is allocated per call.
#include <cuda_runtime.h>

#include "common.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB per device

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array in the current device's context.  It is
// looked up on every call (a host-side query that allocates nothing): a
// cached address could outlive the context it belongs to (after
// cudaDeviceReset, or in another context on the same device).
int scratch_on_current_device(void** ptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return (int)e;
    *ptr = p;
    return 0;
}

}  // namespace

extern "C" int st_attn_fwd_noalloc(const st_layout_t* L, int B, int H, int d, int dtype,
                                   int causal, float scale, const void* q, const void* k,
                                   const void* v, int out_dtype, void* out, float* lse,
                                   void* stream) {
    if (!L) return ST_ERR_NULL;
    if (B < 1 || H < 1 || (int64_t)B * H > 65535) return ST_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ST_ERR_UNSUPPORTED;
    if (dtype != ST_DTYPE_F32 && dtype != ST_DTYPE_BF16) return ST_ERR_UNSUPPORTED;
    const size_t need = st::fwd_workspace_bytes((int64_t)B * L->S * H, d, dtype);
    if (need > kScratchBytes) return ST_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (need > 0) {
        const int e = scratch_on_current_device(&scratch);
        if (e != 0) return st::record_cuda_error(e);
    }
    return st_attn_fwd(L, B, H, d, dtype, causal, scale, q, k, v, out_dtype, out, lse, scratch,
                       need > 0 ? kScratchBytes : 0, stream);
}
