// zg_qk.cuh -- QK RMSNorm + partial RoPE applied to head rows that sit in
// shared memory in the 128-byte-swizzled layout the tensor cores read.
//
// Definition (ZGCM-1-7B 完全解説, gotosocial explainer, section "アーキテクチャ";
// hyper.ai summary of arXiv 2609.13356, section "方法"): queries and keys get
// RMSNorm ("QK normalisation") and partial RoPE with rotary ratio 0.33.
// Readings used here: x_hat = x * (mean_d x^2 + eps)^(-1/2) * w, then dims
// [0, r) rotate in pairs (j, j + r/2) by pos * theta^(-2j/r); dims [r, d) pass.
#pragma once
#include "zg_kernels.cuh"

namespace zg {

// 2*pi split for Cody-Waite range reduction (Cody & Waite, "Software Manual for
// the Elementary Functions", 1980): C1 has 8 significant bits so n * C1 is exact
// for |n| < 2^16; C2 and C3 carry the rest of 2*pi.
constexpr double kTwoPiD = 6.283185307179586476925286766559;
constexpr float kTwoPiC1 = 6.28125f;
constexpr float kTwoPiC2 = float(kTwoPiD - 6.28125);
constexpr float kTwoPiC3 = float(kTwoPiD - 6.28125 - double(float(kTwoPiD - 6.28125)));
constexpr float kInvTwoPi = float(1.0 / kTwoPiD);

// cos / sin of pos * f with f = f_hi + f_lo, for 0 <= pos < 2^24 and pos * f < 4e5.
// The product is carried as a float pair (exact FMA residual), reduced modulo 2*pi
// with the three-part constant, then fed to the hardware sine / cosine on [-pi, pi].
__device__ __forceinline__ void rope_cos_sin(int pos, float f_hi, float f_lo, float& c, float& s) {
    const float p = static_cast<float>(pos);
    const float a_hi = p * f_hi;
    const float a_err = fmaf(p, f_hi, -a_hi);
    const float a_lo = fmaf(p, f_lo, a_err);
    const float n = rintf(a_hi * kInvTwoPi);
    float r = fmaf(-n, kTwoPiC1, a_hi);
    r = fmaf(-n, kTwoPiC2, r);
    r = fmaf(-n, kTwoPiC3, r);
    r += a_lo;
    __sincosf(r, &s, &c);
}

__device__ __forceinline__ float ld_bf16(const uint8_t* p) {
    return __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
}
__device__ __forceinline__ void st_bf16(uint8_t* p, float x) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
}

// Address of element e of row `row` in a tile made of 64-element (128-byte) chunks,
// each chunk a block of rows x 128 B with the 128-byte swizzle, chunk_stride apart.
__device__ __forceinline__ uint8_t* sw_elem(uint8_t* base, uint32_t chunk_stride, int row, int e) {
    return base + (e >> 6) * chunk_stride + sw128_off(row, (e & 63) >> 3) + ((e & 7) << 1);
}

// In-place RMSNorm + partial RoPE of one D-element row held in a swizzled smem tile.
// Only the calling thread touches this row.  w: [D] float weights (global memory).
template <int D>
__device__ __forceinline__ void qk_norm_rope_row(uint8_t* base, uint32_t chunk_stride, int row, const float* __restrict__ w,
                                                 float eps, int pos, const RopeConsts& rc) {
    constexpr int NC = D / 8;  // 16-byte chunks per row
    uint4 v[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c)
        v[c] = *reinterpret_cast<const uint4*>(base + (c >> 3) * chunk_stride + sw128_off(row, c & 7));
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint32_t u[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = bf16lo(u[k]), b = bf16hi(u[k]);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
    }
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    const int r = 2 * rc.half;
    // pass-through dims [r, D): scale now; dims [0, r) stay raw for the rotation pass
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c * 8 + 8 <= r) continue;
        uint32_t u[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = c * 8 + 2 * k;
            float a = bf16lo(u[k]), b = bf16hi(u[k]);
            if (e >= r) a = a * inv * __ldg(w + e);
            if (e + 1 >= r) b = b * inv * __ldg(w + e + 1);
            u[k] = pack_bf16x2(a, b);
        }
        *reinterpret_cast<uint4*>(base + (c >> 3) * chunk_stride + sw128_off(row, c & 7)) =
            make_uint4(u[0], u[1], u[2], u[3]);
    }
    // rotated dims: pairs (j, j + half)
#pragma unroll 1
    for (int j = 0; j < rc.half; ++j) {
        uint8_t* p1 = sw_elem(base, chunk_stride, row, j);
        uint8_t* p2 = sw_elem(base, chunk_stride, row, j + rc.half);
        const float x1 = ld_bf16(p1) * inv * __ldg(w + j);
        const float x2 = ld_bf16(p2) * inv * __ldg(w + j + rc.half);
        float cs, sn;
        rope_cos_sin(pos, rc.f_hi[j], rc.f_lo[j], cs, sn);
        st_bf16(p1, x1 * cs - x2 * sn);
        st_bf16(p2, x2 * cs + x1 * sn);
    }
}

}  // namespace zg
