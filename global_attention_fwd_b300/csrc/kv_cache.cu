// kv_cache.cu -- the decode caches a prefill leaves behind.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ": a local
// (sliding-window) layer keeps the keys and values of the most recent 128 tokens,
// a global layer those of the whole sequence; the decode step reads exactly these
// caches.  Keys are stored as the decode step uses them: normalised and rotated
// (k_hat = RoPE(RMSNorm(k; wk, eps), pos)), rounded to bf16; values are stored raw.
//
// One warp per (sequence b, token i, KV head g) row of the tokens a layer keeps:
//   global layer: every token, slot pos[b, i] of an S-slot cache (0 <= pos < S);
//   local layer:  the last min(L, S) tokens, slot pos[b, i] mod S of an S-slot ring.
// A row whose position has no slot (negative, or >= S in a global cache) is not
// written and is reported in the device error word (code kErrPosition).
// E4M3 caches store e4m3(k_hat * k_scale) and e4m3(v * v_scale), rounded to nearest
// and saturated at the largest finite value.
#include <cuda_fp8.h>

#include "zg_qk.cuh"

namespace zg {
namespace {

template <int D>
__global__ void __launch_bounds__(256) kv_cache_kernel(const __grid_constant__ CacheParams p) {
    __shared__ __align__(16) float buf[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_keep = p.L - p.i0;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // (b, i - i0, g) flattened
    if (row >= static_cast<long long>(p.B) * n_keep * p.Hkv) return;
    const int g = static_cast<int>(row % p.Hkv);
    const long long bt = row / p.Hkv;
    const int b = static_cast<int>(bt / n_keep);
    const int i = p.i0 + static_cast<int>(bt % n_keep);
    const long long src = (static_cast<long long>(b) * p.L + i) * p.Hkv + g;  // row of k / v
    if (!idx_ok(p.ctl, src, static_cast<long long>(p.B) * p.L * p.Hkv, 80)) return;
    const int pos = __ldg(p.pos + static_cast<long long>(b) * p.L + i);
    long long slot;
    if (p.ring) {
        slot = pos >= 0 ? pos % p.S : -1;
    } else {
        slot = (pos >= 0 && pos < p.S) ? pos : -1;
    }
    if (slot < 0) {
        if (lane == 0) report(p.ctl, 80, kErrPosition);
        return;
    }
    const long long dst = ((static_cast<long long>(b) * p.Hkv + g) * p.S + slot) * D;
    if (!idx_ok(p.ctl, dst / D, static_cast<long long>(p.B) * p.Hkv * p.S, 81)) return;
    // the same per-warp arithmetic as the decode step's own cache write (bit-identical keys)
    norm_rope_warp_d<D>(p.k + src * D, p.wk, p.eps, pos, p.rope, 1.0f, buf[warp]);
    for (int e = 2 * lane; e < D; e += 64) {
        const float k0 = buf[warp][e], k1 = buf[warp][e + 1];
        const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162*>(p.v + src * D + e);
        if (p.fp8) {
            const float ks = p.k_scale, vs = p.v_scale;
            *reinterpret_cast<__nv_fp8x2_storage_t*>(reinterpret_cast<uint8_t*>(p.cache_k) + dst + e) =
                __nv_cvt_float2_to_fp8x2(make_float2(k0 * ks, k1 * ks), __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<__nv_fp8x2_storage_t*>(reinterpret_cast<uint8_t*>(p.cache_v) + dst + e) =
                __nv_cvt_float2_to_fp8x2(make_float2(__low2float(vv) * vs, __high2float(vv) * vs), __NV_SATFINITE,
                                         __NV_E4M3);
        } else {
            *reinterpret_cast<uint32_t*>(p.cache_k + dst + e) = pack_bf16x2(k0, k1);
            *reinterpret_cast<__nv_bfloat162*>(p.cache_v + dst + e) = vv;
        }
    }
}

}  // namespace

cudaError_t launch_kv_cache(const CacheParams& p, int d, cudaStream_t s) {
    if (d != 64 && d != 128) return cudaErrorInvalidValue;
    const long long rows = static_cast<long long>(p.B) * (p.L - p.i0) * p.Hkv;
    if (rows <= 0) return cudaSuccess;
    if (d == 128)
        kv_cache_kernel<128><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(p);
    else
        kv_cache_kernel<64><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
