// kv_cache.cu -- the decode caches a prefill leaves behind.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ": a local
// (sliding-window) layer keeps the keys and values of the most recent 128 tokens,
// a global layer those of the whole sequence; the decode step reads exactly these
// caches.  Keys are stored as the decode step uses them: normalised and rotated
// (k_hat = RoPE(RMSNorm(k; wk, eps), pos)), rounded to bf16; values are stored raw.
//
// One (sequence b, token i, KV head g) row of the tokens a layer keeps per warp at a time:
//   global layer: every token, slot pos[b, i] of an S-slot cache (0 <= pos < S);
//   local layer:  the last min(L, S) tokens, slot pos[b, i] mod S of an S-slot ring.
// A row whose position has no slot (negative, or >= S in a global cache) is not
// written and is reported in the device error word (code kErrPosition).
// E4M3 caches store e4m3(k_hat * k_scale) and e4m3(v * v_scale), rounded to nearest
// and saturated at the largest finite value.
#include <cuda_fp8.h>

#include <type_traits>

#include "zg_qk.cuh"

namespace zg {
namespace {

// One warp per kRows consecutive rows: every load of those rows (k, v, positions) is issued
// before the first row is transformed, so each warp keeps kRows x 2 x D x 2 bytes in flight.
constexpr int kRows = 4;

template <int D>
__global__ void __launch_bounds__(256) kv_cache_kernel(const __grid_constant__ CacheParams p) {
    constexpr int PER = D / 32;  // elements per lane
    using Vec = typename std::conditional<PER == 4, uint2, uint32_t>::type;
    __shared__ __align__(16) float buf[8][D];
    __shared__ float rope_f[2][kMaxRotHalf];  // rotation frequencies (head, tail) of this launch
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    stage_rope(p.rope, rope_f[0], rope_f[1]);
    __syncthreads();
    // sequence b = blockIdx.y; rows (i - i0, g) of that sequence in 32-bit arithmetic (the host
    // keeps (L - i0) * Hkv below 2^31)
    const int b = blockIdx.y;
    const unsigned hkv = static_cast<unsigned>(p.Hkv);
    const unsigned n_rows = static_cast<unsigned>(p.L - p.i0) * hkv;
    const unsigned row0 = (blockIdx.x * 8u + warp) * kRows;
    float wv[PER];
    norm_weights_lane<D>(p.wk, wv);
    Vec kraw[kRows], vraw[kRows];
    long long src[kRows];
    int pos[kRows], gh[kRows];
    bool live[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const unsigned row = row0 + r;
        live[r] = row < n_rows;
        src[r] = 0;
        pos[r] = 0;
        gh[r] = 0;
        if (!live[r]) continue;
        gh[r] = static_cast<int>(row % hkv);
        const int i = p.i0 + static_cast<int>(row / hkv);
        src[r] = (static_cast<long long>(b) * p.L + i) * p.Hkv + gh[r];  // row of k / v
        live[r] = idx_ok(p.ctl, src[r], static_cast<long long>(p.B) * p.L * p.Hkv, 80);
        if (!live[r]) continue;
        pos[r] = __ldg(p.pos + static_cast<long long>(b) * p.L + i);
        kraw[r] = *reinterpret_cast<const Vec*>(p.k + src[r] * D + lane * PER);
        vraw[r] = *reinterpret_cast<const Vec*>(p.v + src[r] * D + lane * PER);
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        if (!live[r]) continue;
        long long slot;
        if (p.ring) {  // ring sizes fit 32 bits (the host keeps them to the decode window)
            slot = pos[r] >= 0 ? static_cast<long long>(static_cast<unsigned>(pos[r]) % static_cast<unsigned>(p.S)) : -1;
        } else {
            slot = (pos[r] >= 0 && pos[r] < p.S) ? pos[r] : -1;
        }
        if (slot < 0) {
            if (lane == 0) report(p.ctl, 80, kErrPosition);
            continue;
        }
        const long long dst = ((static_cast<long long>(b) * p.Hkv + gh[r]) * p.S + slot) * D;
        if (!idx_ok(p.ctl, dst / D, static_cast<long long>(p.B) * p.Hkv * p.S, 81)) continue;
        // the same per-warp arithmetic as the decode step's own cache write (bit-identical keys)
        float kv[PER];
        const uint32_t* kw = reinterpret_cast<const uint32_t*>(&kraw[r]);
#pragma unroll
        for (int k = 0; k < PER / 2; ++k) {
            kv[2 * k] = __uint_as_float(kw[k] << 16);
            kv[2 * k + 1] = __uint_as_float(kw[k] & 0xFFFF0000u);
        }
        norm_rope_warp_vals<D>(kv, wv, p.eps, pos[r], p.rope.half, rope_f[0], rope_f[1], 1.0f, buf[warp]);
        float kh[PER];
        if constexpr (PER == 4) {
            const float4 t = *reinterpret_cast<const float4*>(buf[warp] + lane * 4);
            kh[0] = t.x, kh[1] = t.y, kh[2] = t.z, kh[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2*>(buf[warp] + lane * 2);
            kh[0] = t.x, kh[1] = t.y;
        }
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(&vraw[r]);
        if (p.fp8) {
            const float ks = p.k_scale, vs = p.v_scale;
            uint32_t ko = 0u, vo = 0u;
#pragma unroll
            for (int k = 0; k < PER / 2; ++k) {
                const uint32_t k2 = __nv_cvt_float2_to_fp8x2(make_float2(kh[2 * k] * ks, kh[2 * k + 1] * ks),
                                                             __NV_SATFINITE, __NV_E4M3);
                const uint32_t v2 = __nv_cvt_float2_to_fp8x2(
                    make_float2(__uint_as_float(vw[k] << 16) * vs, __uint_as_float(vw[k] & 0xFFFF0000u) * vs),
                    __NV_SATFINITE, __NV_E4M3);
                ko |= k2 << (16 * k);
                vo |= v2 << (16 * k);
            }
            uint8_t* ck = reinterpret_cast<uint8_t*>(p.cache_k) + dst + lane * PER;
            uint8_t* cv = reinterpret_cast<uint8_t*>(p.cache_v) + dst + lane * PER;
            if constexpr (PER == 4) {
                *reinterpret_cast<uint32_t*>(ck) = ko;
                *reinterpret_cast<uint32_t*>(cv) = vo;
            } else {
                *reinterpret_cast<uint16_t*>(ck) = static_cast<uint16_t>(ko);
                *reinterpret_cast<uint16_t*>(cv) = static_cast<uint16_t>(vo);
            }
        } else {
            Vec ko;
            uint32_t* kow = reinterpret_cast<uint32_t*>(&ko);
#pragma unroll
            for (int k = 0; k < PER / 2; ++k) kow[k] = pack_bf16x2(kh[2 * k], kh[2 * k + 1]);
            *reinterpret_cast<Vec*>(p.cache_k + dst + lane * PER) = ko;
            *reinterpret_cast<Vec*>(p.cache_v + dst + lane * PER) = vraw[r];
        }
        __syncwarp();  // buf[warp] is reused by the next row
    }
}

}  // namespace

cudaError_t launch_kv_cache(const CacheParams& p, int d, cudaStream_t s) {
    if (d != 64 && d != 128) return cudaErrorInvalidValue;
    const long long rows = static_cast<long long>(p.L - p.i0) * p.Hkv;  // per sequence
    if (rows <= 0 || p.B <= 0) return cudaSuccess;
    if (rows >= (1ll << 31) || p.B > 65535) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>((rows + 8 * kRows - 1) / (8 * kRows)), static_cast<unsigned>(p.B));
    if (d == 128)
        kv_cache_kernel<128><<<grid, 256, 0, s>>>(p);
    else
        kv_cache_kernel<64><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
