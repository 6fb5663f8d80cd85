// noalloc.cu -- zg_hybrid_decode_noalloc: the hybrid decode step for callers
// that cannot allocate device memory.
//
// zg_hybrid_decode needs a caller-provided scratch workspace for its split-K
// partial results.  Some callers cannot call cudaMalloc to make one: for
// example a plugin running inside a host application whose memory manager owns
// every device allocation and does not lend buffers to plugins, or a serving
// loop that must not allocate while it is answering requests.  This entry
// point gives them the same decode step with the scratch taken from a fixed
// array compiled into the library instead.
//
// The array, kScratchBytes long, lives in device global memory of every GPU
// that loads this library, from the first use until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up (cudaGetSymbolAddress, with the device current) on the first call
// made in a CUDA context and kept for that context; a new context on the same
// device (after cudaDeviceReset, say) gets its own lookup on its first call.
// Make that first call before any stream capture begins.  All calls share the
// one array and it keeps the contents of the last call: the decode kernels
// write every scratch entry they later read, so nothing needs clearing between
// calls, but two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on the array and give wrong results.
#include <cuda.h>

#include <mutex>

#include "../../include/zg_attn.h"
#include "zg_kernels.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(ZG_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
struct Cached {
    unsigned long long ctx_id;  // the context the address belongs to (0 = none yet)
    void* addr;
};
Cached g_cache[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// unique id of the current context (driver entry points looked up once)
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// device address of the array in the current context (looked up once per context)
bool scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx) && ctx != 0;  // none yet before the first runtime call
    std::lock_guard<std::mutex> guard(g_lock);
    if (!have_ctx || g_cache[dev].ctx_id != ctx || !g_cache[dev].addr) {
        void* p = nullptr;
        // the lookup also makes the device's primary context current if nothing was
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return false;
        if (!have_ctx && (!current_context_id(&ctx) || ctx == 0)) return false;
        g_cache[dev].ctx_id = ctx;
        g_cache[dev].addr = p;
    }
    *out = g_cache[dev].addr;
    return true;
}

}  // namespace

extern "C" zg_status zg_hybrid_decode_noalloc(const zg_bf16* q, const zg_bf16* k_new, const zg_bf16* v_new,
                                              const zg_bf16* gate, const int32_t* pos, const float* wq,
                                              const float* wk, const uint8_t* is_global, zg_bf16* k_glob,
                                              zg_bf16* v_glob, zg_bf16* k_ring, zg_bf16* v_ring, zg_bf16* out,
                                              int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window,
                                              int rotary_dim, double theta, float eps, zg_stream stream) {
    // the checks of zg_hybrid_decode come first, so a bad call gets the same status from both
    int NG = 0;
    const int st = zg::hybrid_decode_check(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring,
                                           v_ring, out, NL, B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, 0,
                                           1.0f, 1.0f, &NG);
    if (st != ZG_OK) return static_cast<zg_status>(st);
    if (NL == 0 || B == 0) return ZG_OK;
    const size_t need = zg_hybrid_decode_workspace_bytes(NG, B, Hq, d, S_max);
    if (need > kScratchBytes) return ZG_ERR_WORKSPACE;  // beyond the fixed scratch maximum
    void* scratch = nullptr;
    if (need > 0 && !scratch_address(&scratch)) return ZG_ERR_CUDA;
    return zg_hybrid_decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, out, NL,
                            B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, scratch, need ? kScratchBytes : 0,
                            stream);
}
