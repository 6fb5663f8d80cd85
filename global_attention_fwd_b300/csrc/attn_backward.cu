// attn_backward.cu -- gradients of the attention prefill (gated SWA or global).
//
// The forward ("ZGCM-1-7B 完全解説", gotosocial explainer, section "アーキテクチャ"; the
// pages train the model at 4K, which is what needs these gradients):
//   q_hat = RoPE(q * inv_q * wq, pos), inv_q = (mean(q^2) + eps)^-1/2   (k_hat likewise)
//   p_ij = softmax_j(q_hat_i . k_hat_j / sqrt(d)) over the window j in [i - W + 1, i]
//          (W <= 0: every j <= i, a global layer)
//   A_i = sum_j p_ij v_j;   out_i = A_i * sigmoid(g_i)   (global layer: out_i = A_i)
// Given dout, with c = 1/sqrt(d):
//   dA_i = dout_i * sigmoid(g_i),  dg_i = dout_i * A_i * sigmoid(g_i) (1 - sigmoid(g_i))
//   D_i = dA_i . A_i,  ds_ij = p_ij (dA_i . v_j - D_i)
//   dq_hat_i = c sum_j ds_ij k_hat_j,  dk_hat_j = c sum_(i,h) ds_ij q_hat_i,  dv_j = sum_(i,h) p_ij dA_i
//   then back through RoPE (rotation by -angle) and RMSNorm:
//   dx = inv (w * dy) - inv^3 / d * x * sum(x * w * dy).
// Kernels (one warp per row, four dims per lane, fp32, scores recomputed rather than stored):
//   1. q_hat, k_hat of every row into the workspace;
//   2. per query row: the softmax statistics and A in one online pass, dA, dgate, D, then
//      dq_hat in a second pass over the window;
//   3. per key row: dk_hat and dv over the queries whose window holds the key;
//   4. per q and k row: back through RoPE and RMSNorm.
#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int D = 128;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 ld_bf4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
}
__device__ __forceinline__ float4 axpy4(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

// 1. q_hat and k_hat rows (fp32)
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ BackwardParams p) {
    __shared__ float buf[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (row >= nq + nk) return;
    const bool is_q = row < nq;
    const long long r = is_q ? row : row - nq;
    const long long tok = r / (is_q ? p.Hq : p.Hkv);  // b * L + i
    const int pos = __ldg(p.pos + tok);
    norm_rope_warp(is_q ? p.q + r * D : p.k + r * D, is_q ? p.wq : p.wk, p.eps, pos, p.rope, 1.0f, buf[warp]);
    st4((is_q ? p.qh : p.kh) + r * D + lane * 4, ld4(&buf[warp][lane * 4]));
}

// 2. per query row (b, i, h)
__global__ void __launch_bounds__(256) bwd_query_kernel(const __grid_constant__ BackwardParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // (b, i, h)
    if (row >= static_cast<long long>(p.B) * p.L * p.Hq) return;
    const int h = static_cast<int>(row % p.Hq);
    const long long tok = row / p.Hq;
    const int i = static_cast<int>(tok % p.L);
    const long long b = tok / p.L;
    const int g = h / (p.Hq / p.Hkv);
    const int j0 = p.window > 0 ? max(0, i - p.window + 1) : 0;
    const float c = p.scale;
    const float4 q = ld4(p.qh + row * D + lane * 4);
    auto krow = [&](int j) { return ((b * p.L + j) * p.Hkv + g) * D + lane * 4; };
    // online softmax statistics and A
    float m = -INFINITY, l = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = j0; j <= i; ++j) {
        const float s = warp_sum(dot4(q, ld4(p.kh + krow(j)))) * c;
        const float4 vj = ld_bf4(p.v + krow(j));
        if (s > m) {
            const float r = m == -INFINITY ? 0.f : __expf(m - s);
            l = l * r + 1.f;
            a = axpy4(1.f, vj, make_float4(a.x * r, a.y * r, a.z * r, a.w * r));
            m = s;
        } else {
            const float e = __expf(s - m);
            l += e;
            a = axpy4(e, vj, a);
        }
    }
    const float inv_l = 1.f / l;
    a = make_float4(a.x * inv_l, a.y * inv_l, a.z * inv_l, a.w * inv_l);
    // dA and dgate
    const float4 dout = ld_bf4(p.dout + row * D + lane * 4);
    float4 da = dout;
    if (p.gate) {
        const float4 gv = ld_bf4(p.gate + row * D + lane * 4);
        // sigma and 1 - sigma, both without cancellation
        float s0, s1, s2, s3, c0, c1, c2, c3;
        sigmoid_pair(gv.x, s0, c0);
        sigmoid_pair(gv.y, s1, c1);
        sigmoid_pair(gv.z, s2, c2);
        sigmoid_pair(gv.w, s3, c3);
        da = make_float4(dout.x * s0, dout.y * s1, dout.z * s2, dout.w * s3);
        st4(p.dgate + row * D + lane * 4, make_float4(da.x * a.x * c0, da.y * a.y * c1, da.z * a.z * c2, da.w * a.w * c3));
    }
    const float Dd = warp_sum(dot4(da, a));
    // dq_hat
    float4 dq = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = j0; j <= i; ++j) {
        const float4 kj = ld4(p.kh + krow(j));
        const float s = warp_sum(dot4(q, kj)) * c;
        const float dp = warp_sum(dot4(da, ld_bf4(p.v + krow(j))));
        const float ds = __expf(s - m) * inv_l * (dp - Dd);
        dq = axpy4(c * ds, kj, dq);
    }
    st4(p.dqh + row * D + lane * 4, dq);
    st4(p.da + row * D + lane * 4, da);
    if (lane == 0) {
        p.stat[row * 3 + 0] = m;
        p.stat[row * 3 + 1] = inv_l;
        p.stat[row * 3 + 2] = Dd;
    }
}

// 3. per key row (b, j, g)
__global__ void __launch_bounds__(256) bwd_key_kernel(const __grid_constant__ BackwardParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // (b, j, g)
    if (row >= static_cast<long long>(p.B) * p.L * p.Hkv) return;
    const int g = static_cast<int>(row % p.Hkv);
    const long long tok = row / p.Hkv;
    const int j = static_cast<int>(tok % p.L);
    const long long b = tok / p.L;
    const int G = p.Hq / p.Hkv;
    const int i1 = p.window > 0 ? min(p.L - 1, j + p.window - 1) : p.L - 1;
    const float c = p.scale;
    const float4 kj = ld4(p.kh + row * D + lane * 4);
    const float4 vj = ld_bf4(p.v + row * D + lane * 4);
    float4 dk = make_float4(0.f, 0.f, 0.f, 0.f), dv = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = j; i <= i1; ++i) {
        for (int hh = 0; hh < G; ++hh) {
            const long long qr = (b * p.L + i) * p.Hq + g * G + hh;
            const float4 q = ld4(p.qh + qr * D + lane * 4);
            const float4 da = ld4(p.da + qr * D + lane * 4);
            const float m = p.stat[qr * 3 + 0], inv_l = p.stat[qr * 3 + 1], Dd = p.stat[qr * 3 + 2];
            const float s = warp_sum(dot4(q, kj)) * c;
            const float dp = warp_sum(dot4(da, vj));
            const float pr = __expf(s - m) * inv_l;
            dk = axpy4(c * pr * (dp - Dd), q, dk);
            dv = axpy4(pr, da, dv);
        }
    }
    st4(p.dkh + row * D + lane * 4, dk);
    st4(p.dv + row * D + lane * 4, dv);
}

// 4. back through RoPE and RMSNorm, per q row then per k row
__global__ void __launch_bounds__(256) bwd_norm_rope_kernel(const __grid_constant__ BackwardParams p) {
    __shared__ float buf[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (row >= nq + nk) return;
    const bool is_q = row < nq;
    const long long r = is_q ? row : row - nq;
    const long long tok = r / (is_q ? p.Hq : p.Hkv);
    const int pos = __ldg(p.pos + tok);
    float* dst = buf[warp];
    st4(dst + lane * 4, ld4((is_q ? p.dqh : p.dkh) + r * D + lane * 4));
    __syncwarp();
    // the forward rotated (a, b) -> (a cs - b sn, b cs + a sn); its transpose rotates back
    for (int jj = lane; jj < p.rope.half; jj += 32) {
        float cs, sn;
        rope_cos_sin(pos, p.rope.f_hi[jj], p.rope.f_lo[jj], cs, sn);
        const float d1 = dst[jj], d2 = dst[jj + p.rope.half];
        dst[jj] = d1 * cs + d2 * sn;
        dst[jj + p.rope.half] = d2 * cs - d1 * sn;
    }
    __syncwarp();
    const float4 dy = ld4(dst + lane * 4);
    const float4 x = ld_bf4((is_q ? p.q : p.k) + r * D + lane * 4);
    const float4 w = __ldg(reinterpret_cast<const float4*>((is_q ? p.wq : p.wk) + lane * 4));
    const float ss = warp_sum(dot4(x, x));
    const float inv = ss > 0.f || p.eps > 0.f ? rsqrtf(ss * (1.0f / D) + p.eps) : 0.f;  // as the forward
    const float4 wdy = make_float4(w.x * dy.x, w.y * dy.y, w.z * dy.z, w.w * dy.w);
    const float t = warp_sum(dot4(x, wdy)) * inv * inv * inv * (1.0f / D);
    st4((is_q ? p.dq : p.dk) + r * D + lane * 4,
        make_float4(inv * wdy.x - t * x.x, inv * wdy.y - t * x.y, inv * wdy.z - t * x.z, inv * wdy.w - t * x.w));
}

}  // namespace

size_t backward_workspace_bytes(int B, int L, int Hq, int Hkv) {
    const size_t rq = static_cast<size_t>(B) * L * Hq, rk = static_cast<size_t>(B) * L * Hkv;
    return (rq * D * 3 + rq * 3 + rk * D * 2) * sizeof(float);  // qh, da, dqh, stat, kh, dkh
}

cudaError_t launch_backward(const BackwardParams& p, int d, cudaStream_t s) {
    if (d != D) return cudaErrorInvalidValue;
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    if (nq == 0) return cudaSuccess;
    const unsigned both = static_cast<unsigned>((nq + nk + 7) / 8);
    bwd_prep_kernel<<<both, 256, 0, s>>>(p);
    bwd_query_kernel<<<static_cast<unsigned>((nq + 7) / 8), 256, 0, s>>>(p);
    bwd_key_kernel<<<static_cast<unsigned>((nk + 7) / 8), 256, 0, s>>>(p);
    bwd_norm_rope_kernel<<<both, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
