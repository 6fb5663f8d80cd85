// global_prefill.cu -- ungated full-causal GQA attention prefill (the global
// layers) on sm_103a.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ": 5 of the
// 32 layers attend to the whole context, without the output gate; q and k get
// QK RMSNorm and partial RoPE like the local layers.  For query token i, head h
// (KV head g = h / 4):  A = softmax_j(q_hat . k_hat_j / sqrt(d)) v_j, j = 0..i.
//
// Kernel 1 normalises and rotates every key once (one warp per key row) into
// an fp16 workspace, so the quadratic loop below never repeats that work.
//
// Kernel 2: one CTA owns 2T consecutive tokens of one KV head, as two 128-row
// tiles (T = 128 / G tokens x the G query heads of the group each), Q0 and Q1,
// that share every K_hat / V block of 128 keys; heaviest CTAs (longest key ranges)
// first.  Head sizes 64 and 128; GQA ratios G = 1, 2, 4, 8, 16.
//   warp 0      TMA: both Q tiles, then K_hat / V blocks on two-stage rings.
//   warp 1      MMA (one thread): QK0(0), QK1(0), then per block j
//                 PV0(j), QK0(j+1), PV1(j), QK1(j+1)
//               so the tensor core computes one tile's scores while the other
//               tile's softmax runs.  S_t and P_t share TMEM columns (P packed bf16
//               over S); the MMAs of one thread execute in issue order, so
//               QK_t(j+1) overwrites S_t only after PV_t(j) has read P_t(j).
//   warps 4-7   tile 0: normalise + rotate Q0; per block: scores from TMEM, the
//               running max raised only when a block maximum exceeds it by 8
//               (log2 units), O rescaled in place in TMEM when it moves (after
//               PV0(j-1) has completed), P = exp2(...) in bf16 back to TMEM, row
//               sums of the rounded P; finally O / l -> bf16 -> TMA store.
//   warps 8-11  the same for tile 1.
// TMEM: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// Only blocks that reach past the CTA's first query hold keys beyond a diagonal.
#include <cuda_fp8.h>

#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int BK = 128;               // keys per block
constexpr uint32_t CH = 128 * 128;    // one 64-column chunk of 128 rows (16-bit elements)
constexpr int NBAR = 27;
constexpr float kTau = 8.0f;
constexpr int kThreads = 384;
constexpr int kGroupCt = 128;  // CTAs of one (sequence, KV head) scheduled together on long sequences

template <int D, bool F8 = false, bool SWA = false>
struct Glb {
    static constexpr uint32_t TILE = 128 * D * (F8 ? 1 : 2);  // one 128-row x D tile (16-bit: D/64 chunks)
    static constexpr uint32_t OFF_Q = 0;           // Q0, Q1
    static constexpr uint32_t OFF_K = 2 * TILE;    // 2 stages
    static constexpr uint32_t OFF_V = 4 * TILE;    // 2 stages
    static constexpr uint32_t OFF_G = 6 * TILE;    // SWA: gate / output staging, one bf16 tile per Q tile
    static constexpr uint32_t OFF_BAR = OFF_G + (SWA ? 2 * 128 * D * 2 : 0);
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_R = OFF_MISC + 32;  // E4M3: the rotation frequencies (hi, lo)
    static constexpr uint32_t SMEM = OFF_R + (F8 ? 2 * kMaxRotHalf * 4 : 0);
};

// ---------------------------------------------------------------- kernel 1
template <int D>
__global__ void __launch_bounds__(256) khat_kernel(const __grid_constant__ PrefillParams p) {
    __shared__ __align__(16) float buf[8][D];
    __shared__ float rope_f[2][kMaxRotHalf];
    stage_rope(p.rope, rope_f[0], rope_f[1]);
    __syncthreads();
    constexpr int PER = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // (b, j, g) flattened
    const long long nrows = static_cast<long long>(p.B) * p.L * p.Hkv;
    if (row >= nrows) return;
    const long long tok = row / p.Hkv;  // b * L + j
    if (!idx_ok(p.ctl, tok, static_cast<long long>(p.B) * p.L, 82)) return;
    const int pos = __ldg(p.pos + tok);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.k_raw) + row * D + lane * PER;
    float v[PER], wv[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) v[k] = __bfloat162float(x[k]);
    norm_weights_lane<D>(p.wk, wv);
    norm_rope_warp_vals<D>(v, wv, p.eps, pos, p.rope.half, rope_f[0], rope_f[1], 1.0f, buf[warp]);
    __half* kh = static_cast<__half*>(p.khat) + row * D + lane * PER;
    const float* y = buf[warp] + lane * PER;
    if constexpr (PER == 4)
        *reinterpret_cast<uint2*>(kh) = make_uint2(pack_half2(y[0], y[1]), pack_half2(y[2], y[3]));
    else
        *reinterpret_cast<uint32_t*>(kh) = pack_half2(y[0], y[1]);
}

// ---------------------------------------------------------------- E4M3 variant: pre-passes
// E4M3 (FP8) inputs: q, k, v hold e4m3(x * scale) with per-tensor scales.  The products run on
// tcgen05.mma.kind::f8f6f4: q_hat and k_hat are re-quantised to E4M3 after RMSNorm and RoPE with a
// power-of-two scale that maps their bound sqrt(d) max|w| inside the E4M3 range, P is quantised
// to E4M3, V is used as stored.  Both fp8 operands of every product are K-major: the pre-pass
// writes V transposed, [B, Hkv, d, Lp] (Lp = L rounded up to 16, zero padded).
__device__ __forceinline__ float e4m3_to_f(uint8_t u) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(u), __NV_E4M3);
    return __half2float(__half(h));
}
__device__ __forceinline__ uint8_t f_to_e4m3(float x) {
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
// power-of-two scale s with s * sqrt(D) * max|w| <= 448 (the largest finite E4M3); warp-collective
template <int D>
__device__ __forceinline__ float e4m3_hat_scale(const float* w) {
    float m = 0.f;
    for (int e = threadIdx.x & 31; e < D; e += 32) m = fmaxf(m, fabsf(__ldg(w + e)));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float bound = sqrtf(static_cast<float>(D)) * fmaxf(m, 1e-30f) * 1.001f;
    return exp2f(floorf(log2f(448.f / bound)));
}

// In-place RMSNorm + partial RoPE of one E4M3 row (D = 128 bytes, 128-byte swizzle) of a tile:
// x = stored * dq; out = e4m3(RoPE(RMSNorm(x) * w) * s_out).  One thread per row.
template <int D>
__device__ __forceinline__ void qk_norm_rope_row_e4m3(uint8_t* tile, int row, const float* w, float eps, int pos,
                                                      const RopeConsts& rc, float dq, float s_out) {
    static_assert(D == 128, "one 128-byte swizzle row per head row");
    auto at = [&](int e) { return tile + sw128_off(row, e >> 4) + (e & 15); };
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_off(row, c));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = e4m3_to_f(u[k] & 0xFF), b = e4m3_to_f((u[k] >> 8) & 0xFF);
            const float c2 = e4m3_to_f((u[k] >> 16) & 0xFF), d2 = e4m3_to_f(u[k] >> 24);
            ss = fmaf(a, a, fmaf(b, b, fmaf(c2, c2, fmaf(d2, d2, ss))));
        }
    }
    ss *= dq * dq;
    const float f = (ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f) * dq;
#pragma unroll 1
    for (int j = 0; j < rc.half; ++j) {
        const float a = e4m3_to_f(*at(j)) * f * __ldg(w + j);
        const float c = e4m3_to_f(*at(j + rc.half)) * f * __ldg(w + j + rc.half);
        float cs, sn;
        rope_cos_sin(pos, rc.f_hi[j], rc.f_lo[j], cs, sn);
        *at(j) = f_to_e4m3((a * cs - c * sn) * s_out);
        *at(j + rc.half) = f_to_e4m3((c * cs + a * sn) * s_out);
    }
    // the dims past the rotated ones: whole 16-byte chunks with paired conversions, the rest bytewise
    const int c_first = (2 * rc.half + 15) / 16;  // chunks [c_first, D / 16) hold no rotated dim
    for (int e = 2 * rc.half; e < 16 * c_first; ++e) *at(e) = f_to_e4m3(e4m3_to_f(*at(e)) * f * __ldg(w + e) * s_out);
    const float fs = f * s_out;
#pragma unroll 1
    for (int c = c_first; c < D / 16; ++c) {
        uint4* cp = reinterpret_cast<uint4*>(tile + sw128_off(row, c));
        const uint4 v = *cp;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 w4 = __ldg(reinterpret_cast<const float4*>(w + 16 * c + 4 * k));
            const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] & 0xFFFFu), __NV_E4M3);
            const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] >> 16), __NV_E4M3);
            const float2 x01 = __half22float2(__half2(h01)), x23 = __half22float2(__half2(h23));
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x01.x * fs * w4.x, x01.y * fs * w4.y), __NV_SATFINITE,
                                                         __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x23.x * fs * w4.z, x23.y * fs * w4.w), __NV_SATFINITE,
                                                         __NV_E4M3);
            o[k] = lo | (hi << 16);
        }
        *cp = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// The same with the rotary width 2*HALF compiled in: the chunks holding rotated dims stay in
// registers (no per-element shared-memory round trip), and the SL lanes that share a position (the
// G query heads of a token sit in consecutive rows) split the cos/sin evaluations and exchange them
// with shuffles.  f_hi / f_lo: the rotation frequencies in shared memory (read by lane-dependent
// index).  Every lane of the warp calls it.
template <int D, int SL, int HALF>
__device__ __forceinline__ void qk_norm_rope_row_e4m3_ct(uint8_t* tile, int row, const float* w, float eps, int pos,
                                                         const float* f_hi, const float* f_lo, float dq, float s_out) {
    static_assert(D == 128, "one 128-byte swizzle row per head row");
    constexpr int NR = (2 * HALF + 15) / 16;  // 16-byte chunks holding rotated dims
    static_assert(NR <= D / 16, "rotary width above the head dimension");
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_off(row, c));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a = e4m3_to_f(u[k] & 0xFF), b = e4m3_to_f((u[k] >> 8) & 0xFF);
            const float c2 = e4m3_to_f((u[k] >> 16) & 0xFF), d2 = e4m3_to_f(u[k] >> 24);
            ss = fmaf(a, a, fmaf(b, b, fmaf(c2, c2, fmaf(d2, d2, ss))));
        }
    }
    ss *= dq * dq;
    const float f = (ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f) * dq;
    const float fs = f * s_out;
    // cos/sin: lane (grp | h) evaluates frequencies j = i*SL + h; everyone gathers them below
    const int lane = threadIdx.x & 31;
    const int mine = lane & (SL - 1), grp = lane & ~(SL - 1);
    constexpr int NI = (HALF + SL - 1) / SL;
    float cj[NI], sj[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int jm = i * SL + mine;
        cj[i] = 1.f;
        sj[i] = 0.f;
        if (jm < HALF) rope_cos_sin(pos, f_hi[jm], f_lo[jm], cj[i], sj[i]);
    }
    // the chunks with rotated dims: x * w in registers, rotated, then times f * s_out
    float y[NR * 16];
#pragma unroll
    for (int c = 0; c < NR; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_off(row, c));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 w4 = __ldg(reinterpret_cast<const float4*>(w + 16 * c + 4 * k));
            const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] & 0xFFFFu), __NV_E4M3);
            const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] >> 16), __NV_E4M3);
            const float2 x01 = __half22float2(__half2(h01)), x23 = __half22float2(__half2(h23));
            y[16 * c + 4 * k] = x01.x * w4.x;
            y[16 * c + 4 * k + 1] = x01.y * w4.y;
            y[16 * c + 4 * k + 2] = x23.x * w4.z;
            y[16 * c + 4 * k + 3] = x23.y * w4.w;
        }
    }
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
        const float cs = __shfl_sync(0xffffffffu, cj[j / SL], grp | (j % SL));
        const float sn = __shfl_sync(0xffffffffu, sj[j / SL], grp | (j % SL));
        const float a = y[j], b = y[j + HALF];
        y[j] = a * cs - b * sn;
        y[j + HALF] = b * cs + a * sn;
    }
#pragma unroll
    for (int c = 0; c < NR; ++c) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float* q4 = y + 16 * c + 4 * k;
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(q4[0] * fs, q4[1] * fs), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(q4[2] * fs, q4[3] * fs), __NV_SATFINITE, __NV_E4M3);
            o[k] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(tile + sw128_off(row, c)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    // the chunks past the rotated dims, with paired conversions
#pragma unroll 1
    for (int c = NR; c < D / 16; ++c) {
        uint4* cp = reinterpret_cast<uint4*>(tile + sw128_off(row, c));
        const uint4 v = *cp;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 w4 = __ldg(reinterpret_cast<const float4*>(w + 16 * c + 4 * k));
            const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] & 0xFFFFu), __NV_E4M3);
            const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u[k] >> 16), __NV_E4M3);
            const float2 x01 = __half22float2(__half2(h01)), x23 = __half22float2(__half2(h23));
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x01.x * fs * w4.x, x01.y * fs * w4.y), __NV_SATFINITE,
                                                         __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x23.x * fs * w4.z, x23.y * fs * w4.w), __NV_SATFINITE,
                                                         __NV_E4M3);
            o[k] = lo | (hi << 16);
        }
        *cp = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// k_hat in E4M3 from E4M3 keys, one thread per key row: a CTA stages 128 rows (16 KB) in shared
// memory with coalesced loads (128-byte swizzle), transforms each row in place with the query
// transform's arithmetic (the key weights, the key hat scale), and writes the rows back
// coalesced.  ROT: the rotary width compiled in (then SL lanes, a divisor of Hkv, share a position:
// the KV heads of a token are consecutive rows), or 0 = any width.
template <int D, int SL, int ROT>
__global__ void __launch_bounds__(128) khat_e4m3_kernel(const __grid_constant__ PrefillParams p) {
    static_assert(D == 128, "one 128-byte row per head vector");
    __shared__ __align__(1024) uint8_t tile[128 * D];
    __shared__ float rf[2 * kMaxRotHalf];
    const long long nrows = static_cast<long long>(p.B) * p.L * p.Hkv;
    const long long row0 = static_cast<long long>(blockIdx.x) * 128;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.k_raw);
    uint8_t* dst = reinterpret_cast<uint8_t*>(p.khat);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {  // 16-byte piece i of the CTA's rows: row i / 8, chunk i % 8
        const int i = threadIdx.x + 128 * k, r = i >> 3, c = i & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row0 + r < nrows) v = *reinterpret_cast<const uint4*>(src + (row0 + r) * D + c * 16);
        *reinterpret_cast<uint4*>(tile + sw128_off(r, c)) = v;
    }
    if constexpr (ROT > 0) stage_rope(p.rope, rf, rf + kMaxRotHalf);
    __syncthreads();
    const int r = threadIdx.x;
    const long long row = row0 + r;
    const long long tok = row < nrows ? row / p.Hkv : 0;
    const int pos =
        row < nrows && idx_ok(p.ctl, tok, static_cast<long long>(p.B) * p.L, 94) ? __ldg(p.pos + tok) : 0;
    const float s_kh = e4m3_hat_scale<D>(p.wk);
    if constexpr (ROT > 0)
        qk_norm_rope_row_e4m3_ct<D, SL, ROT / 2>(tile, r, p.wk, p.eps, pos, rf, rf + kMaxRotHalf, p.in_dequant_k,
                                                 s_kh);
    else
        qk_norm_rope_row_e4m3<D>(tile, r, p.wk, p.eps, pos, p.rope, p.in_dequant_k, s_kh);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        const int i = threadIdx.x + 128 * k, rr = i >> 3, c = i & 7;
        if (row0 + rr < nrows)
            *reinterpret_cast<uint4*>(dst + (row0 + rr) * D + c * 16) =
                *reinterpret_cast<const uint4*>(tile + sw128_off(rr, c));
    }
}

template <int D, int ROT>
cudaError_t launch_khat_e4m3(const PrefillParams& p, long long rows, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((rows + 127) / 128);
    if constexpr (ROT == 0) {
        khat_e4m3_kernel<D, 1, 0><<<grid, 128, 0, s>>>(p);
    } else {  // lanes sharing a position: the largest power of two <= 8 dividing Hkv
        if (p.Hkv % 8 == 0)
            khat_e4m3_kernel<D, 8, ROT><<<grid, 128, 0, s>>>(p);
        else if (p.Hkv % 4 == 0)
            khat_e4m3_kernel<D, 4, ROT><<<grid, 128, 0, s>>>(p);
        else if (p.Hkv % 2 == 0)
            khat_e4m3_kernel<D, 2, ROT><<<grid, 128, 0, s>>>(p);
        else
            khat_e4m3_kernel<D, 1, ROT><<<grid, 128, 0, s>>>(p);
    }
    return cudaGetLastError();
}

// V^T in E4M3: [B, Hkv, D, Lp] from [B, L, Hkv, D]; one CTA per 128 keys of one (b, KV head).
// 16-byte loads of the key rows into a 132-byte-stride tile (four 4-byte stores each, on distinct
// banks); then each thread transposes blocks of 4 keys x 4 dims with byte permutes, a warp taking
// 32 keys x 16 dims so that its tile reads hit 32 distinct banks and its stores fill whole 32-byte
// sectors of four V^T rows.
template <int D>
__global__ void __launch_bounds__(256) vt_e4m3_kernel(const __grid_constant__ PrefillParams p, uint8_t* vt, int Lp) {
    static_assert(D == 128, "one 128-byte row per head vector");
    __shared__ uint32_t tile[128][D / 4 + 1];
    const int j0 = blockIdx.x * 128, g = blockIdx.y, b = blockIdx.z;
    const uint8_t* v = reinterpret_cast<const uint8_t*>(p.v_raw);
#pragma unroll
    for (int k = 0; k < 128 * D / 16 / 256; ++k) {  // 16-byte piece i: key row i / 8, piece i % 8
        const int i = threadIdx.x + 256 * k, kr = i >> 3, c = i & 7;
        const int j = j0 + kr;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        const long long src = ((static_cast<long long>(b) * p.L + j) * p.Hkv + g) * D + 16 * c;
        if (j < p.L && idx_ok(p.ctl, src + 15, static_cast<long long>(p.B) * p.L * p.Hkv * D, 66))
            w = *reinterpret_cast<const uint4*>(v + src);
        tile[kr][4 * c] = w.x;
        tile[kr][4 * c + 1] = w.y;
        tile[kr][4 * c + 2] = w.z;
        tile[kr][4 * c + 3] = w.w;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int blk = warp * 4 + k;                        // 32 blocks of 32 keys x 16 dims
        const int k4 = (blk & 3) * 8 + (lane >> 2);          // keys 4 k4 .. 4 k4 + 3
        const int d4 = (blk >> 2) * 4 + (lane & 3);          // dims 4 d4 .. 4 d4 + 3
        const int j = j0 + 4 * k4;
        if (j >= Lp) continue;
        uint32_t w[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) w[r] = tile[4 * k4 + r][d4];
        const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140), t1 = __byte_perm(w[2], w[3], 0x5140);
        const uint32_t t2 = __byte_perm(w[0], w[1], 0x7362), t3 = __byte_perm(w[2], w[3], 0x7362);
        const uint32_t o[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632), __byte_perm(t2, t3, 0x5410),
                               __byte_perm(t2, t3, 0x7632)};  // o[c]: dim 4 d4 + c of the four keys
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const long long dst = ((static_cast<long long>(b) * p.Hkv + g) * D + 4 * d4 + c) * Lp + j;
            if (idx_ok(p.ctl, dst + 3, static_cast<long long>(p.B) * p.Hkv * D * Lp, 67))
                *reinterpret_cast<uint32_t*>(vt + dst) = o[c];
        }
    }
}

// Runs body(it, n) over this CTA's work items: blockIdx.x, + gridDim.x, ... while it returns true
// (persistent CTAs), or blockIdx.x alone; n counts the items done before.
template <bool MANY, class F>
__device__ __forceinline__ void for_items(int n_items, F&& body) {
    if constexpr (MANY) {
        for (int it = static_cast<int>(blockIdx.x), n = 0; it < n_items; it += static_cast<int>(gridDim.x), ++n)
            if (!body(it, n)) break;
    } else {
        (void)n_items;
        body(static_cast<int>(blockIdx.x), 0);
    }
}

// ---------------------------------------------------------------- kernel 2
// F8: E4M3 inputs and products (see the pre-passes above); D = 128 only.
// SWA: the gated sliding-window layer on the same pipeline (used for E4M3 inputs): a CTA visits
// only the key blocks that meet its queries' windows, masks both window edges, and multiplies the
// output by sigmoid(gate) in the epilogue.  Its work items (two Q tiles of one KV head) are short,
// so the CTAs are persistent: one per SM walks items blockIdx.x, + gridDim.x, ...; the TMA warp
// fetches the next item's Q, K_hat / V^T blocks and gate tiles while the current one finishes, and
// the gate tiles have their own staging buffer.  The global layer runs one item per CTA.
// ROT (E4M3): the rotary width compiled into the query transform, or 0 = any width.
template <int D, int G, bool F8, bool SWA = false, int ROT = 0>
__global__ void __launch_bounds__(kThreads, 1) global_attn_kernel(const __grid_constant__ PrefillParams p) {
    constexpr int T = 128 / G;  // tokens per tile
    using C = Glb<D, F8, SWA>;
    constexpr uint32_t TILE = C::TILE, OFF_Q = C::OFF_Q, OFF_K = C::OFF_K, OFF_V = C::OFF_V;
    constexpr uint32_t OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC;
    constexpr int NCH = F8 ? 1 : D / 64;  // TMA boxes per 128-row tile (128-byte box rows)
    static_assert(!F8 || D == 128, "E4M3 rows of 128 bytes");
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bar + 0;
    uint64_t* q_ready = bar + 1;   // [2]
    uint64_t* k_full = bar + 3;    // [2]
    uint64_t* v_full = bar + 5;    // [2]
    uint64_t* k_empty = bar + 7;   // [2]
    uint64_t* v_empty = bar + 9;   // [2]
    uint64_t* s_full = bar + 11;   // [2] per tile
    uint64_t* p_ready = bar + 13;  // [2] per tile
    uint64_t* pv_done = bar + 15;  // [2] per tile
    uint64_t* out_bar = bar + 17;  // [2] per tile: the tile's output is in shared memory
    uint64_t* drain = bar + 19;
    uint64_t* gate_full = bar + 20;  // [2] per tile (SWA): the gate tile is in the staging buffer
    uint64_t* q_empty = bar + 22;    // SWA: the item's score products are complete (Q buffer free)
    uint64_t* stg_free = bar + 23;   // [2] per tile (SWA): the output store has read the staging buffer
    uint64_t* sig_ready = bar + 25;  // [2] per tile (SWA): the staging buffer holds sigmoid(gate)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    float* rf_s = reinterpret_cast<float*>(smem + C::OFF_R);  // E4M3: f_hi [kMaxRotHalf], f_lo [kMaxRotHalf]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbg = p.B * p.Hkv;
    const int n_ct = (p.L + 2 * T - 1) / (2 * T);
    const int n_items = n_ct * nbg;
    // One work item: Q tiles i0 .. i0 + 2T - 1 of KV head g of sequence b, and its key blocks
    // jlo .. jlo + nkb - 1 (both tiles need the same blocks): from 0 for the global layer, from the
    // block of the first key of the first query's window for SWA.
    struct Item {
        int g, b, i0, jlo, nkb;
    };
    auto item = [&](int it) {
        // Heaviest (longest key range) first.  Long sequences: in groups of kGroupCt CTAs of one
        // (b, g), so that the CTAs resident together read the same K_hat / V blocks and share them in L2.
        int ct, bg;
        if (n_ct >= 2 * kGroupCt) {
            const int q = it / (kGroupCt * nbg);  // group, heaviest first
            const int r = it - q * kGroupCt * nbg;
            const int sz = min(kGroupCt, n_ct - q * kGroupCt);
            bg = r / sz;
            ct = n_ct - 1 - (q * kGroupCt + r % sz);
        } else {
            ct = n_ct - 1 - it / nbg;
            bg = it % nbg;
        }
        Item w;
        w.g = bg % p.Hkv;
        w.b = bg / p.Hkv;
        w.i0 = ct * 2 * T;
        w.jlo = SWA ? max(0, w.i0 - p.window + 1) / BK : 0;
        w.nkb = (w.i0 + 2 * T + BK - 1) / BK - w.jlo;
        return w;
    };
    const Item w0 = item(static_cast<int>(blockIdx.x));  // the first (for the global layer, only) item

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 50, kErrAlign);
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&q_ready[i], 128);
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 128);
            mbar_init(&pv_done[i], 1);
            mbar_init(&out_bar[i], 128);
            mbar_init(&gate_full[i], 1);
            mbar_init(&stg_free[i], 1);
            mbar_init(&sig_ready[i], 64);
        }
        mbar_init(q_empty, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if constexpr (F8 && ROT > 0) stage_rope(p.rope, rf_s, rf_s + kMaxRotHalf);
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t sbase = smem_u32(smem);
    auto aborted = [&]() { return *abort_flag != 0; };
    auto fail = [&]() { *abort_flag = 1; };
    // registers: the TMA / MMA warpgroup (warps 0-3) hands most of its share to the two softmax
    // warpgroups, which hold a 128-score row each: 128 x 64 + 256 x 216 <= 384 x 168 (the launch's)
    if (warp < 4) {
        regs_dec<64>();
        if (warp == 0) {
            // ------------------------------------------------------------ TMA
            if (lane == 0 && !aborted()) {
                tma_prefetch_desc(&p.tm_q);
                tma_prefetch_desc(&p.tm_kh);
                tma_prefetch_desc(F8 ? &p.tm_vt : &p.tm_v);
                tma_prefetch_desc(&p.tm_out);
                if constexpr (SWA) tma_prefetch_desc(&p.tm_gate);
                bool ok = true;
                int J = 0;  // key blocks of earlier items: the ring's position
                for_items<SWA>(n_items, [&](int it, int n) {
                    const Item w = n == 0 ? w0 : item(it);
                    // the previous item's score products have read the Q buffer
                    if (SWA && n > 0 && !(ok = mbar_wait(q_empty, (n - 1) & 1, p.ctl, 68))) return false;
                    mbar_arrive_expect_tx(q_full, 2 * TILE);
                    for (int t = 0; t < 2; ++t)
                        for (int ch = 0; ch < NCH; ++ch)
                            tma_load_4d(smem + OFF_Q + t * TILE + ch * CH, &p.tm_q, q_full, ch * 64, w.g * G, w.i0 + t * T, w.b);
                    for (int j = 0; j < w.nkb && ok && !aborted(); ++j) {
                        const int jj = J + j, st = jj & 1;
                        ok = mbar_wait(&k_empty[st], ((jj >> 1) & 1) ^ 1, p.ctl, 51);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&k_full[st], TILE);
                        for (int ch = 0; ch < NCH; ++ch)
                            tma_load_4d(smem + OFF_K + st * TILE + ch * CH, &p.tm_kh, &k_full[st], ch * 64, w.g,
                                        (w.jlo + j) * BK, w.b);
                        ok = mbar_wait(&v_empty[st], ((jj >> 1) & 1) ^ 1, p.ctl, 52);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&v_full[st], TILE);
                        if constexpr (F8)  // V^T block: 128 key bytes per row, D rows
                            tma_load_4d(smem + OFF_V + st * TILE, &p.tm_vt, &v_full[st], (w.jlo + j) * BK, 0, w.g, w.b);
                        else
                            for (int ch = 0; ch < NCH; ++ch)
                                tma_load_4d(smem + OFF_V + st * TILE + ch * CH, &p.tm_v, &v_full[st], ch * 64, w.g,
                                            (w.jlo + j) * BK, w.b);
                    }
                    if constexpr (SWA) {  // the gate tiles (bf16), once the previous item's outputs are stored
                        for (int t = 0; t < 2 && ok && !aborted(); ++t) {
                            if (n > 0 && !(ok = mbar_wait(&stg_free[t], (n - 1) & 1, p.ctl, 69))) break;
                            mbar_arrive_expect_tx(&gate_full[t], (D / 64) * CH);
                            for (int ch = 0; ch < D / 64; ++ch)
                                tma_load_4d(smem + C::OFF_G + t * (D / 64) * CH + ch * CH, &p.tm_gate, &gate_full[t],
                                            ch * 64, w.g * G, w.i0 + t * T, w.b);
                        }
                    }
                    J += w.nkb;
                    return ok && !aborted();
                });
                if (!ok) fail();
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA
            if (lane == 0 && !aborted()) {
                // jj: the key block's place in the ring (counted over this CTA's items); j: within the item
                auto qk = [&](int t, int jj) {
                    constexpr uint32_t idesc = idesc_f16_f32(128, BK, false, false);  // fp16, or E4M3 (code 0)
                    const uint32_t kofs = OFF_K + (jj & 1) * TILE;
                    if constexpr (F8) {
    #pragma unroll
                        for (int ks = 0; ks < D / 32; ++ks)  // 32 E4M3 values = 32 bytes per k-step
                            umma_f8(tbase + t * 128, sdesc(sbase + OFF_Q + t * TILE + ks * 32, 16, 1024, kSw128),
                                    sdesc(sbase + kofs + ks * 32, 16, 1024, kSw128), idesc, ks > 0);
                    } else {
    #pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t co = (ks >> 2) * CH + (ks & 3) * 32;
                            umma_bf16(tbase + t * 128, sdesc(sbase + OFF_Q + t * TILE + co, 16, 1024, kSw128),
                                      sdesc(sbase + kofs + co, 16, 1024, kSw128), idesc, ks > 0);
                        }
                    }
                    umma_commit(&s_full[t]);
                };
                auto pv = [&](int t, int jj, int j) {
                    const uint32_t vofs = OFF_V + (jj & 1) * TILE;
                    if constexpr (F8) {
                        // P (E4M3, four per TMEM column) times V^T (K-major: rows = dims, 128 key bytes each)
                        constexpr uint32_t idesc = idesc_f16_f32(128, D, false, false);
    #pragma unroll
                        for (int ks = 0; ks < BK / 32; ++ks)
                            umma_f8_tmem_a(tbase + 256 + t * 128, tbase + t * 128 + ks * 8,
                                           sdesc(sbase + vofs + ks * 32, 16, 1024, kSw128), idesc,
                                           (j > 0 || ks > 0) ? 1u : 0u);
                    } else {
                        constexpr uint32_t idesc = idesc_bf16_f32(128, D, false, true);
    #pragma unroll
                        for (int ks = 0; ks < BK / 16; ++ks)
                            umma_tmem_a(tbase + 256 + t * 128, tbase + t * 128 + ks * 8,
                                        sdesc(sbase + vofs + ks * 16 * 128, CH, 1024, kSw128), idesc,
                                        (j > 0 || ks > 0) ? 1u : 0u);
                    }
                    umma_commit(&pv_done[t]);
                };
                bool ok = true;
                int J = 0;
                for_items<SWA>(n_items, [&](int it, int n) {
                    const int nkb = n == 0 ? w0.nkb : item(it).nkb;
                    ok = mbar_wait(&q_ready[0], n & 1, p.ctl, 53) && mbar_wait(&q_ready[1], n & 1, p.ctl, 53) &&
                         mbar_wait(&k_full[J & 1], (J >> 1) & 1, p.ctl, 54);
                    if (ok) {
                        tc_fence_after();
                        qk(0, J);
                        qk(1, J);
                        umma_commit(&k_empty[J & 1]);
                        if (SWA && nkb == 1) umma_commit(q_empty);
                    }
                    for (int j = 0; j < nkb && ok && !aborted(); ++j) {
                        const int jj = J + j;
                        const bool more = j + 1 < nkb;
                        ok = mbar_wait(&v_full[jj & 1], (jj >> 1) & 1, p.ctl, 55) && mbar_wait(&p_ready[0], jj & 1, p.ctl, 56);
                        if (!ok) break;
                        tc_fence_after();
                        pv(0, jj, j);
                        if (more) {
                            ok = mbar_wait(&k_full[(jj + 1) & 1], ((jj + 1) >> 1) & 1, p.ctl, 57);
                            if (!ok) break;
                            tc_fence_after();
                            qk(0, jj + 1);
                        }
                        ok = mbar_wait(&p_ready[1], jj & 1, p.ctl, 58);
                        if (!ok) break;
                        tc_fence_after();
                        pv(1, jj, j);
                        umma_commit(&v_empty[jj & 1]);
                        if (more) {
                            qk(1, jj + 1);
                            umma_commit(&k_empty[(jj + 1) & 1]);
                            if (SWA && j + 2 == nkb) umma_commit(q_empty);  // the item's last score products
                        }
                    }
                    J += nkb;
                    return ok && !aborted();
                });
                if (!ok) fail();
                umma_commit(drain);
                (void)mbar_wait(drain, 0, p.ctl, 59);
            }
        } else if constexpr (SWA) {
            // ------------------------------------------------------------ sigmoid(gate) (warps 2, 3)
            // each gate tile, once landed, becomes sigmoid(gate) in place (fp32, rounded to bf16:
            // 2^-9 relative at every magnitude), so that the epilogue only multiplies
            const int tid = static_cast<int>(threadIdx.x) - 64;
            bool ok = true;
            for_items<SWA>(n_items, [&](int, int n) {
                for (int t = 0; t < 2 && ok; ++t) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&gate_full[t], n & 1, p.ctl, 70));
                    if (!ok) break;
                    uint4* g4 = reinterpret_cast<uint4*>(smem + C::OFF_G + t * (D / 64) * CH);
#pragma unroll 4
                    for (int i = tid; i < 128 * D / 8; i += 64) {
                        const uint4 v = g4[i];
                        const float2 a = sigmoid2_f32(bf2f2(v.x)), b = sigmoid2_f32(bf2f2(v.y));
                        const float2 c = sigmoid2_f32(bf2f2(v.z)), d = sigmoid2_f32(bf2f2(v.w));
                        g4[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(b.x, b.y), pack_bf16x2(c.x, c.y),
                                           pack_bf16x2(d.x, d.y));
                    }
                    mbar_arrive(&sig_ready[t]);
                }
                return ok && !aborted();
            });
            if (!ok) fail();
        }
    } else {
        regs_inc<216>();
        // ------------------------------------------------------------ softmax / epilogue
        const int t = (warp - 4) >> 2;            // tile of this warpgroup
        const int row = threadIdx.x - 128 - t * 128;  // tile row = TMEM lane
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_addr + t * 128;
        const uint32_t o_addr = lane_addr + 256 + t * 128;
        uint8_t* qt = smem + OFF_Q + t * TILE;
        const int tt = row / G;
        // E4M3: q_hat and k_hat are stored times power-of-two scales (undone in the score scale)
        const float s_qh = F8 ? e4m3_hat_scale<D>(p.wq) : 1.f;
        const float s_kh = F8 ? e4m3_hat_scale<D>(p.wk) : 1.f;
        const float sc = F8 ? p.scale_log2 / (s_qh * s_kh) : p.scale_log2;
        // the position of this thread's query row in an item
        auto pos_of = [&](const Item& w) {
            const int iq = w.i0 + t * T + tt;
            const long long pi = static_cast<long long>(w.b) * p.L + iq;
            return iq < p.L && idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 83) ? __ldg(p.pos + pi) : 0;
        };
        // q_hat of this thread's row of the n-th item, in place in the Q buffer
        auto q_transform = [&](int n, int pos) {
            const bool okq = __all_sync(0xffffffffu, mbar_wait(q_full, n & 1, p.ctl, 60));
            if (okq) {
                if constexpr (F8 && ROT > 0)
                    qk_norm_rope_row_e4m3_ct<D, G, ROT / 2>(qt, row, p.wq, p.eps, pos, rf_s, rf_s + kMaxRotHalf,
                                                            p.in_dequant_q, s_qh);
                else if constexpr (F8)
                    qk_norm_rope_row_e4m3<D>(qt, row, p.wq, p.eps, pos, p.rope, p.in_dequant_q, s_qh);
                else
                    qk_norm_rope_row<D>(qt, CH, row, p.wq, p.eps, pos, p.rope);
                fence_async_smem();
            }
            mbar_arrive(&q_ready[t]);
            if (!okq) fail();
            return okq;
        };
        bool ok = true;
        int J = 0;
        for_items<SWA>(n_items, [&](int it, int n) {
            const Item w = n == 0 ? w0 : item(it);
            const int g = w.g, b = w.b, i0 = w.i0, jlo = w.jlo, nkb = w.nkb;
            const int iq = i0 + t * T + tt;
            ok = q_transform(n, pos_of(w));
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nkb && ok; ++j) {
                const int jj = J + j;
                if (aborted() || !__all_sync(0xffffffffu, mbar_wait(&s_full[t], jj & 1, p.ctl, 61))) {
                    fail();
                    break;
                }
                tc_fence_after();
                uint32_t r[128];
                tmem_ld32(s_addr + 0, r);
                tmem_ld32(s_addr + 32, r + 32);
                tmem_ld32(s_addr + 64, r + 64);
                tmem_ld32(s_addr + 96, r + 96);
                tmem_wait_ld();
                const int kmax = iq - (jlo + j) * BK;  // last valid key column of this row in the block
                // SWA: the warp's 32 rows are 32 / G consecutive tokens, so most 32-column chunks lie
                // wholly inside or wholly outside all their windows; `dead` marks the outside ones
                // (left out of the maximum, P = 0 without exponentials), and only chunks that hold a
                // window edge of some row are masked element by element
                uint32_t dead = 0;
                if constexpr (SWA) {
                    const int kmin = kmax - p.window + 1;  // first key column inside the window
    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int lo = 32 * c, hi = 32 * c + 31;
                        if (__all_sync(0xffffffffu, lo > kmax || hi < kmin)) {
                            dead |= 1u << c;
                        } else if (__any_sync(0xffffffffu, hi > kmax || lo < kmin)) {
    #pragma unroll
                            for (int k = lo; k <= hi; ++k)
                                if (k > kmax || k < kmin) r[k] = __float_as_uint(-INFINITY);
                        }
                    }
                } else if ((jlo + j + 1) * BK - 1 > i0) {  // the block reaches past the CTA's first query
    #pragma unroll
                    for (int k = 0; k < 128; ++k)
                        if (k > kmax) r[k] = __float_as_uint(-INFINITY);
                }
                // block maximum: eight independent chains of three-input maxima, then their maximum
                float a8[8];
                if constexpr (SWA) {
    #pragma unroll
                    for (int i = 0; i < 8; ++i) a8[i] = -INFINITY;
    #pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if ((dead >> c) & 1u) continue;
    #pragma unroll
                        for (int k = 32 * c; k < 32 * c + 32; k += 16)
    #pragma unroll
                            for (int i = 0; i < 8; ++i)
                                a8[i] = fmax3(a8[i], __uint_as_float(r[k + i]), __uint_as_float(r[k + 8 + i]));
                    }
                } else {
    #pragma unroll
                    for (int i = 0; i < 8; ++i) a8[i] = fmaxf(__uint_as_float(r[i]), __uint_as_float(r[i + 8]));
    #pragma unroll
                    for (int k = 16; k < 128; k += 16)
    #pragma unroll
                        for (int i = 0; i < 8; ++i) a8[i] = fmax3(a8[i], __uint_as_float(r[k + i]), __uint_as_float(r[k + 8 + i]));
                }
                const float mx = fmaxf(fmax3(fmax3(a8[0], a8[1], a8[2]), a8[3], a8[4]), fmax3(a8[5], a8[6], a8[7]));
                const float mb = mx * sc;
                float m_new = m_run;
                if (m_run == -INFINITY || mb > m_run + kTau) m_new = mb;
                const float corr = m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new);
                if (j > 0 && __any_sync(0xffffffffu, m_new != m_run)) {
                    // O(j-1) must be complete before it is scaled in place
                    if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[t], (jj - 1) & 1, p.ctl, 62))) {
                        fail();
                        break;
                    }
                    tc_fence_after();
    #pragma unroll 1
                    for (int cb = 0; cb < D; cb += 32) {
                        uint32_t o[32];
                        tmem_ld32(o_addr + cb, o);
                        tmem_wait_ld();
    #pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
                        tmem_st32(o_addr + cb, o);
                    }
                    tmem_wait_st();
                }
                l_run *= corr;
                m_run = m_new;
                // a row whose window has not begun yet (SWA) has m_run = -inf and every score masked: P = 0
                const float m_exp = m_run == -INFINITY ? 0.f : m_run;
                const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(-m_exp, -m_exp);
                float2 l2 = make_float2(0.f, 0.f), l3 = make_float2(0.f, 0.f);
    #pragma unroll
                for (int cb = 0; cb < 128; cb += 32) {
                    if (SWA && ((dead >> (cb / 32)) & 1u)) {  // outside every row's window: P = 0
                        uint32_t z[16] = {};
                        if constexpr (F8)
                            tmem_st8(s_addr + cb / 4, z);
                        else
                            tmem_st16(s_addr + cb / 2, z);
                        continue;
                    }
                    if constexpr (F8) {
                        // P in E4M3 (at most 2^8 with the lazy maximum: inside the range), four per column.
                        // The row sums add the rounded values the product uses: 16 per fp16 lane (at most
                        // 2^12, so in range; relative rounding <= 9 * 2^-11, far below P's own 2^-4), then
                        // once per 32 columns into fp32.
                        uint32_t pk[8];
                        __half2 hacc = __float2half2_rn(0.f);
    #pragma unroll
                        for (int k = 0; k < 32; k += 4) {
                            const float2 x0 = fma2(make_float2(__uint_as_float(r[cb + k]), __uint_as_float(r[cb + k + 1])), sc2, nm2);
                            const float2 x1 = fma2(make_float2(__uint_as_float(r[cb + k + 2]), __uint_as_float(r[cb + k + 3])), sc2, nm2);
                            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                                make_float2(ex2_approx(x0.x), ex2_approx(x0.y)), __NV_SATFINITE, __NV_E4M3);
                            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                                make_float2(ex2_approx(x1.x), ex2_approx(x1.y)), __NV_SATFINITE, __NV_E4M3);
                            pk[k / 4] = uint32_t(lo) | (uint32_t(hi) << 16);
                            const __half2_raw hl = __nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3);
                            const __half2_raw hh = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
                            hacc = __hadd2(hacc, __hadd2(__half2(hl), __half2(hh)));
                        }
                        l2 = add2(l2, __half22float2(hacc));
                        tmem_st8(s_addr + cb / 4, pk);  // P over S (these columns are already in registers)
                    } else {
                        uint32_t pk[16];
    #pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const float2 x = fma2(make_float2(__uint_as_float(r[cb + k]), __uint_as_float(r[cb + k + 1])), sc2, nm2);
                            pk[k / 2] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
                            if (k & 2)
                                acc_bf16x2(pk[k / 2], l3.x, l3.y);
                            else
                                acc_bf16x2(pk[k / 2], l2.x, l2.y);
                        }
                        tmem_st16(s_addr + cb / 2, pk);  // P over S (these columns are already in registers)
                    }
                }
                l_run += (l2.x + l2.y) + (l3.x + l3.y);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_ready[t]);
            }
            // ---- epilogue: O / l -> bf16 -> staging tile -> TMA store.  The staging tile is the tile's
            // Q buffer, or (E4M3, whose Q buffer is half the size of the bf16 output) the K stages for
            // tile 0 and the V stages for tile 1, free once the tile's last product has completed; SWA:
            // the gate tile, turned into sigmoid(gate) by warps 2 and 3, which the output overwrites in place.
            uint8_t* stg = SWA ? smem + C::OFF_G + t * (D / 64) * CH : F8 ? smem + (t == 0 ? OFF_K : OFF_V) : qt;
            if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (J + nkb - 1) & 1, p.ctl, 63));
            if (SWA && ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(&sig_ready[t], n & 1, p.ctl, 65));
            if (ok) {
                tc_fence_after();
                const float inv_l = l_run > 0.f ? (F8 ? p.in_dequant_v : 1.0f) / l_run : 0.f;
    #pragma unroll 1
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + cb, o);
                    tmem_wait_ld();
    #pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t ou[4];
                        const int e0 = cb + q4 * 8;
                        uint4* dst = reinterpret_cast<uint4*>(stg + (e0 >> 6) * CH + sw128_off(row, (e0 & 63) >> 3));
                        if constexpr (SWA) {  // out = A * sigmoid(gate), sigmoid(gate) read from the same place
                            const uint4 gv = *dst;
                            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    #pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float2 sg = bf2f2(gw[k]);
                                ou[k] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * k]) * inv_l * sg.x,
                                                    __uint_as_float(o[q4 * 8 + 2 * k + 1]) * inv_l * sg.y);
                            }
                        } else {
    #pragma unroll
                            for (int k = 0; k < 4; ++k)
                                ou[k] = pack_bf16x2(__uint_as_float(o[q4 * 8 + 2 * k]) * inv_l,
                                                    __uint_as_float(o[q4 * 8 + 2 * k + 1]) * inv_l);
                        }
                        *dst = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                    }
                }
                fence_async_smem();
            }
            tc_fence_before();
            mbar_arrive(&out_bar[t]);
            if (row == 0 && ok) {
                if (!mbar_wait(&out_bar[t], n & 1, p.ctl, 64)) {
                    fail();
                } else if (i0 + t * T < p.L) {  // a tile that starts past the end has nothing to store
                    for (int ch = 0; ch < D / 64; ++ch)
                        tma_store_4d(&p.tm_out, stg + ch * CH, ch * 64, g * G, i0 + t * T, b);
                    bulk_commit();
                    if constexpr (SWA)
                        bulk_wait_read_all();  // the next gate tile may land once the store has read this one
                    else
                        bulk_wait_all();
                }
                if (SWA) mbar_arrive(&stg_free[t]);
            }
            if (!ok) fail();
            J += nkb;
            return ok && !aborted();
        });
        if constexpr (SWA)  // the outputs' stores complete before the CTA exits
            if (row == 0) bulk_wait_all();
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        // abandoned tile: give copies still in flight time to land before memory is released
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D, int G, bool F8, bool SWA, int ROT>
cudaError_t launch_t(const PrefillParams& p, cudaStream_t s) {
    constexpr int T = 128 / G;
    const long long rows = static_cast<long long>(p.B) * p.L * p.Hkv;
    if constexpr (F8) {
        const cudaError_t ek = launch_khat_e4m3<D, ROT>(p, rows, s);
        if (ek != cudaSuccess) return ek;
        const dim3 vg(static_cast<unsigned>((p.vt_lp + 127) / 128), static_cast<unsigned>(p.Hkv),
                      static_cast<unsigned>(p.B));
        vt_e4m3_kernel<D><<<vg, 256, 0, s>>>(p, p.vt_ws, p.vt_lp);
    } else {
        khat_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(p);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto k = global_attn_kernel<D, G, F8, SWA, ROT>;
    constexpr uint32_t smem = Glb<D, F8, SWA>::SMEM;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    long long ctas = static_cast<long long>(p.B) * p.Hkv * ((p.L + 2 * T - 1) / (2 * T));
    if constexpr (SWA) {  // persistent: one CTA per SM
        int dev = 0, sms = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        ctas = ctas < sms ? ctas : sms;
    }
    k<<<static_cast<unsigned>(ctas), kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D, bool F8, bool SWA = false, int ROT = 0>
cudaError_t launch_d(const PrefillParams& p, cudaStream_t s) {
    switch (p.Hq / p.Hkv) {
        case 1: return launch_t<D, 1, F8, SWA, ROT>(p, s);
        case 2: return launch_t<D, 2, F8, SWA, ROT>(p, s);
        case 4: return launch_t<D, 4, F8, SWA, ROT>(p, s);
        case 8: return launch_t<D, 8, F8, SWA, ROT>(p, s);
        case 16: return launch_t<D, 16, F8, SWA, ROT>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool global_supports(int d, int G) { return (d == 64 || d == 128) && (G == 1 || G == 2 || G == 4 || G == 8 || G == 16); }
int global_q_tile_tokens(int G) { return 128 / G; }

cudaError_t launch_global_prefill(const PrefillParams& p, int d, cudaStream_t s) {
    if (p.Hkv <= 0 || p.Hq % p.Hkv || !global_supports(d, p.Hq / p.Hkv)) return cudaErrorInvalidValue;
    // E4M3: the ZGCM-1 rotary width (42 of 128 dims) compiled in, any other through the general transform
    constexpr int kRot = 42;
    if (p.fp8 && p.swa) {
        if (d != 128 || p.window < 1) return cudaErrorInvalidValue;
        return 2 * p.rope.half == kRot ? launch_d<128, true, true, kRot>(p, s) : launch_d<128, true, true>(p, s);
    }
    if (p.fp8) {
        if (d != 128) return cudaErrorInvalidValue;
        return 2 * p.rope.half == kRot ? launch_d<128, true, false, kRot>(p, s) : launch_d<128, true>(p, s);
    }
    return d == 128 ? launch_d<128, false>(p, s) : launch_d<64, false>(p, s);
}

}  // namespace zg
