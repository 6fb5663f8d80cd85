// zg_qk.cuh -- QK RMSNorm + partial RoPE applied to head rows that sit in
// shared memory in the 128-byte-swizzled layout the tensor cores read.
//
// Definition (ZGCM-1-7B 完全解説, gotosocial explainer, section "アーキテクチャ";
// hyper.ai summary of arXiv 2609.13356, section "方法"): queries and keys get
// RMSNorm ("QK normalisation") and partial RoPE with rotary ratio 0.33.
// Readings used here: x_hat = x * (mean_d x^2 + eps)^(-1/2) * w, then dims
// [0, r) rotate in pairs (j, j + r/2) by pos * theta^(-2j/r); dims [r, d) pass.
#pragma once
#include <cuda_fp16.h>

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
// Reads bf16, writes fp16: RMSNorm bounds every element of x_hat by sqrt(D) * max|w|
// (x_i^2 <= sum x^2 = D * rms^2, and RoPE preserves the norm of each pair), so fp16
// holds q_hat / k_hat with 3 more mantissa bits than bf16 for any |w| < 4096.
// Only the calling thread touches this row.  w: [D] float weights (global memory).
template <int D>
__device__ __forceinline__ void qk_norm_rope_row(uint8_t* base, uint32_t chunk_stride, int row, const float* __restrict__ w,
                                                 float eps, int pos, const RopeConsts& rc) {
    constexpr int NC = D / 8;  // 16-byte chunks per row
    // pass 0: sum of squares, streaming the row chunk by chunk (keeps register use low)
    float ss = 0.f;
#pragma unroll 4
    for (int c = 0; c < NC; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(base + (c >> 3) * chunk_stride + sw128_off(row, c & 7));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = bf16lo(u[k]), b = bf16hi(u[k]);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
    }
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    // pass 1: y = x * inv * w for every dim, stored as fp16
#pragma unroll 4
    for (int c = 0; c < NC; ++c) {
        uint8_t* cp = base + (c >> 3) * chunk_stride + sw128_off(row, c & 7);
        const uint4 v = *reinterpret_cast<const uint4*>(cp);
        uint32_t u[4] = {v.x, v.y, v.z, v.w};
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + c * 8));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + c * 8 + 4));
        const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            u[k] = pack_half2(bf16lo(u[k]) * inv * ww[2 * k], bf16hi(u[k]) * inv * ww[2 * k + 1]);
        *reinterpret_cast<uint4*>(cp) = make_uint4(u[0], u[1], u[2], u[3]);
    }
    // pass 2: rotate the pairs (j, j + half) of the normalised values
#pragma unroll 1
    for (int j = 0; j < rc.half; ++j) {
        __half* p1 = reinterpret_cast<__half*>(sw_elem(base, chunk_stride, row, j));
        __half* p2 = reinterpret_cast<__half*>(sw_elem(base, chunk_stride, row, j + rc.half));
        const float x1 = __half2float(*p1), x2 = __half2float(*p2);
        float cs, sn;
        rope_cos_sin(pos, rc.f_hi[j], rc.f_lo[j], cs, sn);
        *p1 = __float2half_rn(x1 * cs - x2 * sn);
        *p2 = __float2half_rn(x2 * cs + x1 * sn);
    }
}

// In-place RMSNorm + partial RoPE of one row of a swizzled smem tile with TWO lanes per
// row: lanes 2i and 2i+1 of the warp own the same row, the even lane the first half of
// the D values and the odd lane the second half.  SL (a power of two >= 2) consecutive
// lanes share one RoPE position (SL = 2 for key rows, 2G for the G query heads of a
// token): each lane evaluates cos/sin for every SL-th frequency and they exchange them
// with shuffles; the even lane of each row applies the rotations.  Every lane of the
// warp must call this, with the same half.  w_s: the D weights, f_hi / f_lo: the rotation
// frequencies, both in shared memory (read by lane-dependent index, which the kernel parameter
// space would serve one address at a time).
template <int D, int SL>
__device__ __forceinline__ void qk_norm_rope_row_pair(uint8_t* base, uint32_t chunk_stride, int row, const float* w_s,
                                                      float eps, int pos, int half, const float* f_hi,
                                                      const float* f_lo, bool active = true) {
    constexpr int NC2 = D / 16;  // 16-byte chunks per half row
    const int lane = threadIdx.x & 31;
    const int part = lane & 1;
    const int c0 = part * NC2;
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = c0; c < c0 + NC2; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(base + (c >> 3) * chunk_stride + sw128_off(row, c & 7));
        const float2 a = bf2f2(v.x), b = bf2f2(v.y), cc = bf2f2(v.z), d = bf2f2(v.w);
        ss2 = fma2(a, a, ss2);
        ss2 = fma2(b, b, ss2);
        ss2 = fma2(cc, cc, ss2);
        ss2 = fma2(d, d, ss2);
    }
    float ss = ss2.x + ss2.y;
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int c = c0; c < c0 + NC2; ++c) {
        uint8_t* cp = base + (c >> 3) * chunk_stride + sw128_off(row, c & 7);
        const uint4 v = *reinterpret_cast<const uint4*>(cp);
        const float4 w0 = *reinterpret_cast<const float4*>(w_s + c * 8);
        const float4 w1 = *reinterpret_cast<const float4*>(w_s + c * 8 + 4);
        const float2 y0 = mul2(mul2(bf2f2(v.x), make_float2(w0.x, w0.y)), inv2);
        const float2 y1 = mul2(mul2(bf2f2(v.y), make_float2(w0.z, w0.w)), inv2);
        const float2 y2 = mul2(mul2(bf2f2(v.z), make_float2(w1.x, w1.y)), inv2);
        const float2 y3 = mul2(mul2(bf2f2(v.w), make_float2(w1.z, w1.w)), inv2);
        if (active)
            *reinterpret_cast<uint4*>(cp) = make_uint4(pack_half2(y0.x, y0.y), pack_half2(y1.x, y1.y),
                                                       pack_half2(y2.x, y2.y), pack_half2(y3.x, y3.y));
    }
    __syncwarp();  // the odd lane's half is in shared memory before the even lane rotates
    const int mine = lane & (SL - 1);
    const int grp = lane & ~(SL - 1);
    constexpr int NI = (kMaxRotHalf + SL - 1) / SL;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        if (i * SL >= half) break;  // uniform over the warp
        const int jm = i * SL + mine;
        float cs = 1.f, sn = 0.f;
        if (jm < half) rope_cos_sin(pos, f_hi[jm], f_lo[jm], cs, sn);
#pragma unroll
        for (int h = 0; h < SL; ++h) {
            const float c2 = __shfl_sync(0xffffffffu, cs, grp | h);
            const float s2 = __shfl_sync(0xffffffffu, sn, grp | h);
            const int j = i * SL + h;
            if (active && part == 0 && j < half) {
                __half* p1 = reinterpret_cast<__half*>(sw_elem(base, chunk_stride, row, j));
                __half* p2 = reinterpret_cast<__half*>(sw_elem(base, chunk_stride, row, j + half));
                const float x1 = __half2float(*p1), x2 = __half2float(*p2);
                *p1 = __float2half_rn(x1 * c2 - x2 * s2);
                *p2 = __float2half_rn(x2 * c2 + x1 * s2);
            }
        }
    }
}

// As qk_norm_rope_row_pair, for a rotary width 2*HALF known at compile time: the even
// lane keeps the first ceil(2*HALF/8) chunks of its half row in registers and rotates
// them there, so no per-element shared-memory round trip is needed.
template <int D, int SL, int HALF>
__device__ __forceinline__ void qk_norm_rope_row_pair_ct(uint8_t* base, uint32_t chunk_stride, int row,
                                                         const float* w_s, float eps, int pos, const float* f_hi,
                                                         const float* f_lo, bool active = true) {
    constexpr int NC2 = D / 16;
    constexpr int NR = (2 * HALF + 7) / 8;  // chunks holding rotated dims
    static_assert(NR <= NC2, "rotated dims must lie in the first half row");
    const int lane = threadIdx.x & 31;
    const int part = lane & 1;
    const int c0 = part * NC2;
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int c = 0; c < NC2; ++c) {
        const uint4 v =
            *reinterpret_cast<const uint4*>(base + ((c0 + c) >> 3) * chunk_stride + sw128_off(row, (c0 + c) & 7));
        const float2 a = bf2f2(v.x), b = bf2f2(v.y), cc = bf2f2(v.z), d = bf2f2(v.w);
        ss2 = fma2(a, a, ss2);
        ss2 = fma2(b, b, ss2);
        ss2 = fma2(cc, cc, ss2);
        ss2 = fma2(d, d, ss2);
    }
    float ss = ss2.x + ss2.y;
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    const float2 inv2 = make_float2(inv, inv);
    float y[NR * 8];  // even lane: normalised dims [0, 8*NR) before rotation
    // chunk c of this lane's half row: x * inv * w (kept for the rotation on the even lane's first NR
    // chunks, stored otherwise)
    auto chunk = [&](int c, float2 (&yy)[4]) {
        const int cg = c0 + c;
        const uint4 v = *reinterpret_cast<const uint4*>(base + (cg >> 3) * chunk_stride + sw128_off(row, cg & 7));
        const float4 w0 = *reinterpret_cast<const float4*>(w_s + cg * 8);
        const float4 w1 = *reinterpret_cast<const float4*>(w_s + cg * 8 + 4);
        yy[0] = mul2(mul2(bf2f2(v.x), make_float2(w0.x, w0.y)), inv2);
        yy[1] = mul2(mul2(bf2f2(v.y), make_float2(w0.z, w0.w)), inv2);
        yy[2] = mul2(mul2(bf2f2(v.z), make_float2(w1.x, w1.y)), inv2);
        yy[3] = mul2(mul2(bf2f2(v.w), make_float2(w1.z, w1.w)), inv2);
    };
    auto store = [&](int c, const float2 (&yy)[4]) {
        const int cg = c0 + c;
        *reinterpret_cast<uint4*>(base + (cg >> 3) * chunk_stride + sw128_off(row, cg & 7)) =
            make_uint4(pack_half2(yy[0].x, yy[0].y), pack_half2(yy[1].x, yy[1].y), pack_half2(yy[2].x, yy[2].y),
                       pack_half2(yy[3].x, yy[3].y));
    };
#pragma unroll
    for (int c = 0; c < NR; ++c) {
        float2 yy[4];
        chunk(c, yy);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[c * 8 + 2 * k] = yy[k].x;
            y[c * 8 + 2 * k + 1] = yy[k].y;
        }
        if (active && part == 1) store(c, yy);
    }
#pragma unroll 1  // rolled: this helper runs beside the kernel's other roles, and code size costs fetch
    for (int c = NR; c < NC2; ++c) {  // no rotated dims here (on either lane)
        float2 yy[4];
        chunk(c, yy);
        if (active) store(c, yy);
    }
    // cos/sin: lane (grp | h) evaluates frequencies j = i*SL + h; everyone gathers them
    const int mine = lane & (SL - 1);
    const int grp = lane & ~(SL - 1);
    constexpr int NI = (HALF + SL - 1) / SL;
    float cj[NI], sj[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int jm = i * SL + mine;
        cj[i] = 1.f;
        sj[i] = 0.f;
        if (jm < HALF) rope_cos_sin(pos, f_hi[jm], f_lo[jm], cj[i], sj[i]);
    }
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
        const float cs = __shfl_sync(0xffffffffu, cj[j / SL], grp | (j % SL));
        const float sn = __shfl_sync(0xffffffffu, sj[j / SL], grp | (j % SL));
        const float a = y[j], b = y[j + HALF];
        y[j] = a * cs - b * sn;
        y[j + HALF] = b * cs + a * sn;
    }
    if (active && part == 0) {
#pragma unroll
        for (int c = 0; c < NR; ++c)
            *reinterpret_cast<uint4*>(base + (c >> 3) * chunk_stride + sw128_off(row, c & 7)) =
                make_uint4(pack_half2(y[c * 8 + 0], y[c * 8 + 1]), pack_half2(y[c * 8 + 2], y[c * 8 + 3]),
                           pack_half2(y[c * 8 + 4], y[c * 8 + 5]), pack_half2(y[c * 8 + 6], y[c * 8 + 7]));
    }
}

// RMSNorm + partial RoPE of one D-element head vector with one warp; lane l holds elements
// l*D/32 .. l*D/32 + D/32 - 1 in v (fp32); the result times `scale` goes to dst[D] (fp32, shared
// memory).  The decode step and the cache writer both use it, so a key cached by a prefill and
// one cached by a decode step agree bit for bit.
// The rotation frequencies come as pointers (f_hi[j], f_lo[j], j < half): a kernel that runs this
// for many rows stages them in shared memory, because lane j reading element j straight from the
// kernel parameters is a divergent constant-bank access, served one address at a time.
template <int D>
__device__ __forceinline__ void norm_rope_warp_vals(const float (&v)[D / 32], const float (&wv)[D / 32], float eps,
                                                    int pos, int half, const float* f_hi, const float* f_lo,
                                                    float scale, float* dst) {
    constexpr int PER = D / 32;
    static_assert(PER == 2 || PER == 4, "head sizes 64 and 128");
    const int lane = threadIdx.x & 31;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) ss = fmaf(v[k], v[k], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    float o4[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) o4[k] = v[k] * inv * wv[k];
    if constexpr (PER == 4)  // one vector store per lane: no bank conflicts
        *reinterpret_cast<float4*>(dst + lane * 4) = make_float4(o4[0], o4[1], o4[2], o4[3]);
    else
        *reinterpret_cast<float2*>(dst + lane * 2) = make_float2(o4[0], o4[1]);
    __syncwarp();
    for (int j = lane; j < half; j += 32) {
        const float a = dst[j], b = dst[j + half];
        float cs, sn;
        rope_cos_sin(pos, f_hi[j], f_lo[j], cs, sn);
        dst[j] = a * cs - b * sn;
        dst[j + half] = b * cs + a * sn;
    }
    __syncwarp();
    if (scale != 1.0f)
        for (int e = lane; e < D; e += 32) dst[e] *= scale;
    __syncwarp();
}
// Copy the rotation frequencies of a launch into shared memory; every thread of the block calls
// it, and a __syncthreads() follows before they are read.
__device__ __forceinline__ void stage_rope(const RopeConsts& rc, float* s_hi, float* s_lo) {
    for (int j = threadIdx.x; j < rc.half; j += blockDim.x) {
        s_hi[j] = rc.f_hi[j];
        s_lo[j] = rc.f_lo[j];
    }
}
// the weights of lane l's elements, for norm_rope_warp_vals
template <int D>
__device__ __forceinline__ void norm_weights_lane(const float* w, float (&wv)[D / 32]) {
#pragma unroll
    for (int k = 0; k < D / 32; ++k) wv[k] = __ldg(w + (threadIdx.x & 31) * (D / 32) + k);
}
// the same with x (bf16) read from global memory
template <int D>
__device__ __forceinline__ void norm_rope_warp_d(const __nv_bfloat16* x, const float* w, float eps, int pos,
                                                 const RopeConsts& rc, float scale, float* dst) {
    float v[D / 32], wv[D / 32];
#pragma unroll
    for (int k = 0; k < D / 32; ++k) v[k] = __bfloat162float(x[(threadIdx.x & 31) * (D / 32) + k]);
    norm_weights_lane<D>(w, wv);
    norm_rope_warp_vals<D>(v, wv, eps, pos, rc.half, rc.f_hi, rc.f_lo, scale, dst);
}

// RMSNorm + partial RoPE of one 128-element head vector with one warp; x is bf16 in global memory.
// Result (fp32, times `scale`) goes to smem dst[128].
__device__ __forceinline__ void norm_rope_warp(const __nv_bfloat16* x, const float* w, float eps, int pos, const RopeConsts& rc,
                               float scale, float* dst) {
    const int lane = threadIdx.x & 31;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + lane * 4);
    float v[4] = {bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y)};
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / 128) + eps) : 0.f;
    const float4 ww = __ldg(reinterpret_cast<const float4*>(w + lane * 4));
    dst[lane * 4 + 0] = v[0] * inv * ww.x;
    dst[lane * 4 + 1] = v[1] * inv * ww.y;
    dst[lane * 4 + 2] = v[2] * inv * ww.z;
    dst[lane * 4 + 3] = v[3] * inv * ww.w;
    __syncwarp();
    for (int j = lane; j < rc.half; j += 32) {
        const float a = dst[j], b = dst[j + rc.half];
        float cs, sn;
        rope_cos_sin(pos, rc.f_hi[j], rc.f_lo[j], cs, sn);
        dst[j] = a * cs - b * sn;
        dst[j + rc.half] = b * cs + a * sn;
    }
    __syncwarp();
    if (scale != 1.0f)
        for (int e = lane; e < 128; e += 32) dst[e] *= scale;
    __syncwarp();
}

}  // namespace zg
