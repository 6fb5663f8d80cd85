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
// that loads this library, from the first use until the process exits.  Its
// device address is looked up once per device (cudaGetSymbolAddress, with that
// device current) on the first call made on that device; make that first call
// before any stream capture begins.  All calls share the one array and it keeps
// the contents of the last call: the decode kernels write every scratch entry
// they later read, so nothing needs clearing between calls, but two calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on the array and give wrong results.
#include <mutex>

#include "../../include/zg_attn.h"

namespace {

constexpr size_t kScratchBytes = size_t(ZG_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {};

// device address of the array on the current device (looked up once per device)
bool scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return false;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return true;
}

}  // namespace

extern "C" zg_status zg_hybrid_decode_noalloc(const zg_bf16* q, const zg_bf16* k_new, const zg_bf16* v_new,
                                              const zg_bf16* gate, const int32_t* pos, const float* wq,
                                              const float* wk, const uint8_t* is_global, zg_bf16* k_glob,
                                              zg_bf16* v_glob, zg_bf16* k_ring, zg_bf16* v_ring, zg_bf16* out,
                                              int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window,
                                              int rotary_dim, double theta, float eps, zg_stream stream) {
    if (!is_global) return ZG_ERR_NULL;
    int NG = 0;
    for (int l = 0; l < NL; ++l) NG += is_global[l] ? 1 : 0;
    const size_t need = zg_hybrid_decode_workspace_bytes(NG, B, Hq, d, S_max);
    if (need > kScratchBytes) return ZG_ERR_WORKSPACE;  // beyond the fixed scratch maximum
    void* scratch = nullptr;
    if (need > 0 && !scratch_address(&scratch)) return ZG_ERR_CUDA;
    return zg_hybrid_decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, out, NL,
                            B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, scratch, need ? kScratchBytes : 0,
                            stream);
}
