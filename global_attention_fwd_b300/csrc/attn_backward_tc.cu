// attn_backward_tc.cu -- gradients of the windowed attention prefill on the tensor cores
// (sm_103a: tcgen05 MMAs with TMEM accumulators, operands staged by TMA).
//
// The same gradients as attn_backward.cu ("ZGCM-1-7B 完全解説", gotosocial explainer,
// section "アーキテクチャ": QK RMSNorm, partial RoPE, 128-token window including the
// token itself, sigmoid output gate), for the ZGCM-1 shape: d = 128, four query heads
// per KV head, window W <= 128.  With c = 1/sqrt(d), P = softmax(c Q_hat K_hat^T) over
// the window, A = P V:
//   dP = dA V^T,  D = rowsum(dA * A),  dS = P * (dP - D),
//   dQ_hat = c dS K_hat,  dK_hat = c dS^T Q_hat,  dV = P^T dA.
// All MMA operands are bf16 (q_hat, k_hat, dA, P, dS), accumulation fp32.
//
// Kernel 1 (prep, one warp per row): q_hat, k_hat and dA = dout * sigmoid(gate) in bf16.
//
// Kernel 2 (query pass): one CTA per tile of 32 tokens x the 4 query heads of one KV
// head (128 rows); the tile sees the 160 keys [t0 - 128, t0 + 32).
//   warp 4 (one thread): TMA of Q_hat, dA, K_hat, V; the MMAs
//     S = Q_hat K_hat^T  (N = 160)  -> TMEM [0, 160)
//     dP = dA V^T        (N = 160)  -> TMEM [160, 320)
//     O = P V   (P from TMEM, packed over S)          -> TMEM [320, 448)
//     dQ_hat = dS K_hat  (dS from TMEM, packed over dP) -> TMEM [320, 448) (after O is read)
//   warps 0-3 (thread = row = TMEM lane): exact row max and sum over the window, P
//   (unnormalised, bf16) over S; A = O / l, D, dgate = dA * A * (1 - sigmoid(gate)) and
//   the row statistics (max, 1 / l, D) for kernel 3; dS over dP; finally dQ_hat back
//   through RoPE and RMSNorm into dq (fp32).
//
// Kernel 3 (key pass): one CTA per 128 keys of one KV head; the queries that see them
// are the tokens [j0, j0 + 128 + W - 1), visited as query tiles of 32 tokens x 4 heads
// whose Q_hat / dA arrive on a two-stage TMA ring.
//   warp 4: S^T = K_hat Q_hat^T -> [0, 128), dP^T = V dA^T -> [128, 256), then
//     dV += P^T dA -> [256, 384), dK_hat += dS^T Q_hat -> [384, 512)
//     (P^T, dS^T from TMEM, packed over S^T and dP^T; one thread's MMAs run in issue
//     order, so the next tile's S^T overwrites P^T only after dV has read it).
//   warps 0-3 (thread = key row): P^T and dS^T from the row statistics of kernel 2;
//   at the end dV (fp32) and dK_hat back through RoPE and RMSNorm into dk.
#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int D = 128;
constexpr int G = 4;
constexpr int T = 32;                       // tokens per query tile (T * G = 128 rows)
constexpr int NKQ = T + 128;                // keys a query tile sees
constexpr int BK = 128;                     // keys per key tile
constexpr uint32_t CH128 = 128 * 128;       // one 64-column chunk of 128 rows (bf16)
constexpr uint32_t CH160 = NKQ * 128;       // one 64-column chunk of 160 rows
constexpr uint32_t TILE128 = 2 * CH128;
constexpr uint32_t TILE160 = 2 * CH160;
constexpr int SROW = D + 1;                 // staging row stride in floats (conflict-free per-row access)
constexpr uint32_t STAGE = 128 * SROW * 4;  // one staged 128-row fp32 tile
constexpr int kThreads = 160;               // warps 0-3 rows, warp 4 TMA + MMA

// query pass shared memory
constexpr uint32_t QP_Q = 0;
constexpr uint32_t QP_DA = QP_Q + TILE128;
constexpr uint32_t QP_K = QP_DA + TILE128;
constexpr uint32_t QP_V = QP_K + TILE160;
constexpr uint32_t QP_W = QP_V + TILE160;
constexpr uint32_t QP_BAR = QP_W + D * 4;
constexpr uint32_t QP_MISC = QP_BAR + 8 * 8;
constexpr uint32_t QP_SMEM = QP_MISC + 32;
static_assert(STAGE <= QP_W, "the dq staging tile reuses the operand tiles");
static_assert(QP_K % 1024 == 0 && QP_V % 1024 == 0, "128-byte swizzle atoms");

// key pass shared memory
constexpr uint32_t KP_K = 0;
constexpr uint32_t KP_V = KP_K + TILE128;
constexpr uint32_t KP_QD = KP_V + TILE128;      // 2 stages x (Q_hat, dA)
constexpr uint32_t KP_STAT = KP_QD + 4 * TILE128;  // 4 warps x 128 float4
constexpr uint32_t KP_W = KP_STAT + 4 * 128 * 16;
constexpr uint32_t KP_BAR = KP_W + D * 4;
constexpr uint32_t KP_MISC = KP_BAR + 12 * 8;
constexpr uint32_t KP_SMEM = KP_MISC + 32;
static_assert(STAGE <= 4 * TILE128, "the dk / dv staging tile reuses the query ring");
static_assert(KP_SMEM <= 227 * 1024, "shared memory");

// One row held by one thread in a staging row: dy (the gradient of x_hat) in, the gradient
// of the raw row x out.  RoPE rotated (a, b) by +angle, so its transpose rotates by -angle;
// RMSNorm x_hat = x * inv * w with inv = (mean x^2 + eps)^-1/2 gives
// dx = inv * w * dy - inv^3 / d * x * sum(x * w * dy).
__device__ __forceinline__ void row_norm_rope_bwd(float* st, const __nv_bfloat16* __restrict__ x, const float* w_s,
                                                  float eps, int pos, const RopeConsts& rc) {
    for (int j = 0; j < rc.half; ++j) {
        float cs, sn;
        rope_cos_sin(pos, rc.f_hi[j], rc.f_lo[j], cs, sn);
        const float a = st[j], bb = st[j + rc.half];
        st[j] = a * cs + bb * sn;
        st[j + rc.half] = bb * cs - a * sn;
    }
    float ss = 0.f, tw = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; c += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + c);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x0 = bf16lo(w4[e]), x1 = bf16hi(w4[e]);
            ss = fmaf(x0, x0, fmaf(x1, x1, ss));
            tw = fmaf(x0 * w_s[c + 2 * e], st[c + 2 * e], fmaf(x1 * w_s[c + 2 * e + 1], st[c + 2 * e + 1], tw));
        }
    }
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    const float coef = inv * inv * inv * tw * (1.0f / D);
#pragma unroll 4
    for (int c = 0; c < D; c += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(x + c);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            st[c + 2 * e] = inv * w_s[c + 2 * e] * st[c + 2 * e] - coef * bf16lo(w4[e]);
            st[c + 2 * e + 1] = inv * w_s[c + 2 * e + 1] * st[c + 2 * e + 1] - coef * bf16hi(w4[e]);
        }
    }
}

// ---------------------------------------------------------------- kernel 1
__global__ void __launch_bounds__(256) bwd_tc_prep_kernel(const __grid_constant__ BackwardTcParams p) {
    __shared__ float buf[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (row >= nq + nk) return;
    const bool is_q = row < nq;
    const long long r = is_q ? row : row - nq;
    const long long tok = r / (is_q ? p.Hq : p.Hkv);
    const int pos = __ldg(p.pos + tok);
    norm_rope_warp(is_q ? p.q + r * D : p.k + r * D, is_q ? p.wq : p.wk, p.eps, pos, p.rope, 1.0f, buf[warp]);
    const float4 v = *reinterpret_cast<const float4*>(&buf[warp][lane * 4]);
    *reinterpret_cast<uint2*>((is_q ? p.qh : p.kh) + r * D + lane * 4) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    if (is_q && p.gate) {
        const uint2 go = *reinterpret_cast<const uint2*>(p.gate + r * D + lane * 4);
        const uint2 dd = *reinterpret_cast<const uint2*>(p.dout + r * D + lane * 4);
        auto sg = [](float x) { return 1.0f / (1.0f + __expf(-x)); };
        *reinterpret_cast<uint2*>(p.da + r * D + lane * 4) =
            make_uint2(pack_bf16x2(bf16lo(dd.x) * sg(bf16lo(go.x)), bf16hi(dd.x) * sg(bf16hi(go.x))),
                       pack_bf16x2(bf16lo(dd.y) * sg(bf16lo(go.y)), bf16hi(dd.y) * sg(bf16hi(go.y))));
    }
}

// warp-cooperative store of the 32 staged rows of this warp: row r goes to dst(r) when valid(r)
template <class Dst>
__device__ __forceinline__ void store_rows(const float* stage, int warp, int lane, Dst dst) {
    __syncwarp();
    for (int rr = 0; rr < 32; ++rr) {
        const int r = warp * 32 + rr;
        float* d = dst(r);
        if (d) {
            const float* s = stage + r * SROW + lane * 4;
            *reinterpret_cast<float4*>(d + lane * 4) = make_float4(s[0], s[1], s[2], s[3]);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- kernel 2: query pass
__global__ void __launch_bounds__(kThreads, 1) bwd_qpass_kernel(const __grid_constant__ BackwardTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + QP_BAR);
    uint64_t* ld_full = bar + 0;
    uint64_t* s_full = bar + 1;
    uint64_t* p_ready = bar + 2;
    uint64_t* o_full = bar + 3;
    uint64_t* ds_ready = bar + 4;
    uint64_t* dq_full = bar + 5;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + QP_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + QP_MISC + 4);
    float* w_s = reinterpret_cast<float*>(smem + QP_W);
    constexpr uint32_t C_S = 0, C_DP = NKQ, C_O = 2 * NKQ;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbg = p.B * p.Hkv;
    const int t0 = static_cast<int>(blockIdx.x / nbg) * T;
    const int g = static_cast<int>(blockIdx.x % nbg) % p.Hkv;
    const int b = static_cast<int>(blockIdx.x % nbg) / p.Hkv;

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 100, kErrAlign);
        mbar_init(ld_full, 1);
        mbar_init(s_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(o_full, 1);
        mbar_init(ds_ready, 128);
        mbar_init(dq_full, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32)
        *reinterpret_cast<float4*>(w_s + lane * 4) = __ldg(reinterpret_cast<const float4*>(p.wq + lane * 4));
    if (warp == 4) {
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

    if (warp == 4) {
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_qh);
            tma_prefetch_desc(&p.tm_da);
            tma_prefetch_desc(&p.tm_kq);
            tma_prefetch_desc(&p.tm_vq);
            mbar_arrive_expect_tx(ld_full, 2 * TILE128 + 2 * TILE160);
            for (int ch = 0; ch < 2; ++ch) {
                tma_load_4d(smem + QP_Q + ch * CH128, &p.tm_qh, ld_full, ch * 64, g * G, t0, b);
                tma_load_4d(smem + QP_DA + ch * CH128, &p.tm_da, ld_full, ch * 64, g * G, t0, b);
                tma_load_4d(smem + QP_K + ch * CH160, &p.tm_kq, ld_full, ch * 64, g, t0 - 128, b);
                tma_load_4d(smem + QP_V + ch * CH160, &p.tm_vq, ld_full, ch * 64, g, t0 - 128, b);
            }
            constexpr uint32_t id_s = idesc_bf16_f32(128, NKQ, false, false);
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, false, true);
            bool ok = mbar_wait(ld_full, 0, p.ctl, 101);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    const uint32_t ck = (ks >> 2) * CH160 + (ks & 3) * 32;
                    umma_bf16(tbase + C_S, sdesc(sbase + QP_Q + co, 16, 1024, kSw128),
                              sdesc(sbase + QP_K + ck, 16, 1024, kSw128), id_s, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    const uint32_t ck = (ks >> 2) * CH160 + (ks & 3) * 32;
                    umma_bf16(tbase + C_DP, sdesc(sbase + QP_DA + co, 16, 1024, kSw128),
                              sdesc(sbase + QP_V + ck, 16, 1024, kSw128), id_s, ks > 0);
                }
                umma_commit(s_full);
                ok = mbar_wait(p_ready, 0, p.ctl, 102);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < NKQ / 16; ++ks)
                    umma_tmem_a(tbase + C_O, tbase + C_S + ks * 8,
                                sdesc(sbase + QP_V + ks * 16 * 128, CH160, 1024, kSw128), id_o, ks > 0);
                umma_commit(o_full);
                ok = mbar_wait(ds_ready, 0, p.ctl, 103);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < NKQ / 16; ++ks)
                    umma_tmem_a(tbase + C_O, tbase + C_DP + ks * 8,
                                sdesc(sbase + QP_K + ks * 16 * 128, CH160, 1024, kSw128), id_o, ks > 0);
                umma_commit(dq_full);
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ rows (thread = row = TMEM lane)
        const int row = threadIdx.x;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
        const int tt = row / G;
        const int t = t0 + tt;
        const bool valid_row = t < p.L;
        const long long qrow = (static_cast<long long>(b) * p.L + t) * p.Hq + g * G + row % G;
        const int lo = max(128 - t0, tt + 128 - p.window + 1);  // key columns [lo, hi] are in the window
        const int hi = tt + 128;
        const float sl = p.scale_log2;
        bool ok = __all_sync(0xffffffffu, mbar_wait(s_full, 0, p.ctl, 104));
        float m = 0.f, l = 0.f;
        if (ok) {
            tc_fence_after();
            float mx = -INFINITY;
#pragma unroll 1
            for (int k = 0; k < NKQ / 32; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_S + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = 32 * k + i;
                    if (c >= lo && c <= hi) mx = fmaxf(mx, __uint_as_float(r[i]));
                }
            }
            m = (valid_row && mx > -INFINITY) ? mx * sl : 0.f;
#pragma unroll 1
            for (int k = 0; k < NKQ / 32; ++k) {
                uint32_t r[32], pk[16];
                tmem_ld32(lane_addr + C_S + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const int c = 32 * k + i;
                    const bool v0 = valid_row && c >= lo && c <= hi, v1 = valid_row && c + 1 >= lo && c + 1 <= hi;
                    const float e0 = v0 ? ex2_approx(fmaf(__uint_as_float(r[i]), sl, -m)) : 0.f;
                    const float e1 = v1 ? ex2_approx(fmaf(__uint_as_float(r[i + 1]), sl, -m)) : 0.f;
                    pk[i / 2] = pack_bf16x2(e0, e1);
                    const float2 f = bf2f2(pk[i / 2]);  // the sum of the rounded values the MMA uses
                    l += f.x + f.y;
                }
                tmem_st16(lane_addr + C_S + 16 * k, pk);  // P over S: these columns are already read
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_ready);
        if (!ok) fail();
        const float il = l > 0.f ? 1.0f / l : 0.f;
        // ---- A = O / l, D = dA . A, dgate
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(o_full, 0, p.ctl, 105));
        float Dd = 0.f;
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_O + 32 * k, r);
                tmem_wait_ld();
                if (valid_row) {
                    const __nv_bfloat16* dop = p.dout + qrow * D + 32 * k;
#pragma unroll
                    for (int v8 = 0; v8 < 4; ++v8) {
                        const uint4 du = *reinterpret_cast<const uint4*>(dop + 8 * v8);
                        const uint32_t dw[4] = {du.x, du.y, du.z, du.w};
                        float dg[8];
                        if (p.gate) {
                            const uint4 gu = *reinterpret_cast<const uint4*>(p.gate + qrow * D + 32 * k + 8 * v8);
                            const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float gv = (e & 1) ? bf16hi(gw[e / 2]) : bf16lo(gw[e / 2]);
                                const float sg = 1.0f / (1.0f + __expf(-gv));
                                const float a = __uint_as_float(r[8 * v8 + e]) * il;
                                const float dav = ((e & 1) ? bf16hi(dw[e / 2]) : bf16lo(dw[e / 2])) * sg;
                                // D from the bf16 dA the dP product used (the same rounding as the
                                // prep kernel), so that sum_j dS_ij = 0 holds to fp32 rounding
                                Dd = fmaf(__bfloat162float(__float2bfloat16_rn(dav)), a, Dd);
                                dg[e] = dav * a * (1.0f - sg);
                            }
                            float* dgp = p.dgate + qrow * D + 32 * k + 8 * v8;
                            *reinterpret_cast<float4*>(dgp) = make_float4(dg[0], dg[1], dg[2], dg[3]);
                            *reinterpret_cast<float4*>(dgp + 4) = make_float4(dg[4], dg[5], dg[6], dg[7]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float a = __uint_as_float(r[8 * v8 + e]) * il;
                                Dd = fmaf((e & 1) ? bf16hi(dw[e / 2]) : bf16lo(dw[e / 2]), a, Dd);
                            }
                        }
                    }
                }
            }
            if (valid_row) p.stat[qrow] = make_float4(m, il, Dd, 0.f);
            // ---- dS = P (dP - D), packed bf16 over dP
#pragma unroll 1
            for (int k = 0; k < NKQ / 32; ++k) {
                uint32_t pr[16], r[32], dk16[16];
                tmem_ld16(lane_addr + C_S + 16 * k, pr);
                tmem_ld32(lane_addr + C_DP + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 pp = bf2f2(pr[i]);
                    dk16[i] = pack_bf16x2(pp.x * il * (__uint_as_float(r[2 * i]) - Dd),
                                          pp.y * il * (__uint_as_float(r[2 * i + 1]) - Dd));
                }
                tmem_st16(lane_addr + C_DP + 16 * k, dk16);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(ds_ready);
        if (!ok) fail();
        // ---- dq: dQ_hat * c back through RoPE and RMSNorm
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(dq_full, 0, p.ctl, 106));
        if (ok) {
            tc_fence_after();
            float* st = reinterpret_cast<float*>(smem) + row * SROW;  // operand tiles are free now
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_O + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) st[32 * k + i] = __uint_as_float(r[i]) * p.scale;
            }
            if (valid_row)
                row_norm_rope_bwd(st, p.q + qrow * D, w_s, p.eps, __ldg(p.pos + static_cast<long long>(b) * p.L + t),
                                  p.rope);
            store_rows(reinterpret_cast<const float*>(smem), warp, lane, [&](int r) -> float* {
                const int tr = t0 + r / G;
                return tr < p.L ? p.dq + ((static_cast<long long>(b) * p.L + tr) * p.Hq + g * G + r % G) * D : nullptr;
            });
        }
        if (!ok) fail();
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        // abandoned tile: give copies still in flight time to land before memory is released
        const long long c0 = clock64();
        while (clock64() - c0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------- kernel 3: key pass
__global__ void __launch_bounds__(kThreads, 1) bwd_kpass_kernel(const __grid_constant__ BackwardTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + KP_BAR);
    uint64_t* kv_full = bar + 0;
    uint64_t* qd_full = bar + 1;   // [2]
    uint64_t* qd_empty = bar + 3;  // [2]
    uint64_t* s_full = bar + 5;
    uint64_t* p_ready = bar + 6;
    uint64_t* done = bar + 7;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + KP_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + KP_MISC + 4);
    float* w_s = reinterpret_cast<float*>(smem + KP_W);
    float4* stat_s = reinterpret_cast<float4*>(smem + KP_STAT);  // [4 warps][128]
    constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 384;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbg = p.B * p.Hkv;
    const int j0 = static_cast<int>(blockIdx.x / nbg) * BK;
    const int g = static_cast<int>(blockIdx.x % nbg) % p.Hkv;
    const int b = static_cast<int>(blockIdx.x % nbg) / p.Hkv;
    const int u_end = min(p.L, j0 + BK + p.window - 1);  // queries [j0, u_end) see these keys
    const int n_tiles = (u_end - j0 + T - 1) / T;

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 110, kErrAlign);
        mbar_init(kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qd_full[i], 1);
            mbar_init(&qd_empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_ready, 128);
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32)
        *reinterpret_cast<float4*>(w_s + lane * 4) = __ldg(reinterpret_cast<const float4*>(p.wk + lane * 4));
    if (warp == 4) {
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

    if (warp == 4) {
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_qh);
            tma_prefetch_desc(&p.tm_da);
            tma_prefetch_desc(&p.tm_kk);
            tma_prefetch_desc(&p.tm_vk);
            mbar_arrive_expect_tx(kv_full, 2 * TILE128);
            for (int ch = 0; ch < 2; ++ch) {
                tma_load_4d(smem + KP_K + ch * CH128, &p.tm_kk, kv_full, ch * 64, g, j0, b);
                tma_load_4d(smem + KP_V + ch * CH128, &p.tm_vk, kv_full, ch * 64, g, j0, b);
            }
            auto load_qd = [&](int n) {
                const int st = n & 1;
                uint8_t* dst = smem + KP_QD + st * 2 * TILE128;
                mbar_arrive_expect_tx(&qd_full[st], 2 * TILE128);
                for (int ch = 0; ch < 2; ++ch) {
                    tma_load_4d(dst + ch * CH128, &p.tm_qh, &qd_full[st], ch * 64, g * G, j0 + n * T, b);
                    tma_load_4d(dst + TILE128 + ch * CH128, &p.tm_da, &qd_full[st], ch * 64, g * G, j0 + n * T, b);
                }
            };
            constexpr uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, false, true);
            auto issue_s = [&](int n) {  // S^T and dP^T of query tile n
                const uint32_t qd = KP_QD + (n & 1) * 2 * TILE128;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_S, sdesc(sbase + KP_K + co, 16, 1024, kSw128),
                              sdesc(sbase + qd + co, 16, 1024, kSw128), id_s, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_DP, sdesc(sbase + KP_V + co, 16, 1024, kSw128),
                              sdesc(sbase + qd + TILE128 + co, 16, 1024, kSw128), id_s, ks > 0);
                }
                umma_commit(s_full);
            };
            auto issue_acc = [&](int n) {  // dV += P^T dA, dK_hat += dS^T Q_hat
                const uint32_t qd = KP_QD + (n & 1) * 2 * TILE128;
#pragma unroll
                for (int ks = 0; ks < 128 / 16; ++ks) {
                    umma_tmem_a(tbase + C_DV, tbase + C_S + ks * 8,
                                sdesc(sbase + qd + TILE128 + ks * 16 * 128, CH128, 1024, kSw128), id_o,
                                (n > 0 || ks > 0) ? 1u : 0u);
                    umma_tmem_a(tbase + C_DK, tbase + C_DP + ks * 8, sdesc(sbase + qd + ks * 16 * 128, CH128, 1024, kSw128),
                                id_o, (n > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&qd_empty[n & 1]);
            };
            load_qd(0);
            if (n_tiles > 1) load_qd(1);
            bool ok = mbar_wait(kv_full, 0, p.ctl, 111) && mbar_wait(&qd_full[0], 0, p.ctl, 112);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int n = 0; n < n_tiles && ok && !aborted(); ++n) {
                ok = mbar_wait(p_ready, n & 1, p.ctl, 113);
                if (!ok) break;
                tc_fence_after();
                issue_acc(n);
                if (n + 1 < n_tiles) {
                    ok = mbar_wait(&qd_full[(n + 1) & 1], ((n + 1) >> 1) & 1, p.ctl, 114);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(n + 1);
                }
                if (n + 2 < n_tiles) {
                    ok = mbar_wait(&qd_empty[n & 1], (n >> 1) & 1, p.ctl, 115);
                    if (!ok) break;
                    load_qd(n + 2);
                }
            }
            umma_commit(done);
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ rows (thread = key row = TMEM lane)
        const int row = threadIdx.x;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
        const int kj = j0 + row;
        const bool valid_key = kj < p.L;
        const float sl = p.scale_log2;
        const int W = p.window;
        bool ok = true;
        for (int n = 0; n < n_tiles && ok; ++n) {
            const int u0 = j0 + n * T;
            // this tile's query-row statistics, one copy per warp (no barrier across warps:
            // a warp that gives up on a wait must not leave the others blocked)
            float4* sts = stat_s + warp * 128;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = lane + 32 * i;
                const int u = u0 + c / G;
                sts[c] = u < p.L ? p.stat[(static_cast<long long>(b) * p.L + u) * p.Hq + g * G + c % G]
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncwarp();
            if (aborted() || !__all_sync(0xffffffffu, mbar_wait(s_full, n & 1, p.ctl, 116))) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < 128 / 32; ++k) {
                uint32_t r[32], dp[32], pp[16], dd[16];
                tmem_ld32(lane_addr + C_S + 32 * k, r);
                tmem_ld32(lane_addr + C_DP + 32 * k, dp);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float pv[2], dv2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 32 * k + i + e;
                        const int u = u0 + c / G;
                        const float4 s4 = sts[c];
                        const bool v = valid_key && u >= kj && u - kj < W && u < p.L;
                        const float pr = v ? ex2_approx(fmaf(__uint_as_float(r[i + e]), sl, -s4.x)) * s4.y : 0.f;
                        pv[e] = pr;
                        dv2[e] = pr * (__uint_as_float(dp[i + e]) - s4.z);
                    }
                    pp[i / 2] = pack_bf16x2(pv[0], pv[1]);
                    dd[i / 2] = pack_bf16x2(dv2[0], dv2[1]);
                }
                tmem_st16(lane_addr + C_S + 16 * k, pp);   // P^T over S^T
                tmem_st16(lane_addr + C_DP + 16 * k, dd);  // dS^T over dP^T
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_ready);
        }
        if (!ok) fail();
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(done, 0, p.ctl, 117));
        if (ok) {
            tc_fence_after();
            float* stage = reinterpret_cast<float*>(smem + KP_QD);  // the query ring is free now
            float* st = stage + row * SROW;
            const int L = p.L, Hkv = p.Hkv;
            const long long row0 = (static_cast<long long>(b) * L + j0) * Hkv + g;  // (b, j0, g)
            auto dst = [=](float* base) {
                return [=](int r) -> float* { return j0 + r < L ? base + (row0 + static_cast<long long>(r) * Hkv) * D : nullptr; };
            };
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_DV + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) st[32 * k + i] = __uint_as_float(r[i]);
            }
            store_rows(stage, warp, lane, dst(p.dv));
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_DK + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) st[32 * k + i] = __uint_as_float(r[i]) * p.scale;
            }
            if (valid_key)
                row_norm_rope_bwd(st, p.k + ((static_cast<long long>(b) * p.L + kj) * p.Hkv + g) * D, w_s, p.eps,
                                  __ldg(p.pos + static_cast<long long>(b) * p.L + kj), p.rope);
            store_rows(stage, warp, lane, dst(p.dk));
        }
        if (!ok) fail();
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        const long long c0 = clock64();
        while (clock64() - c0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tbase, 512);
}

}  // namespace

bool backward_tc_supports(int d, int Hq, int Hkv, int window) {
    return d == D && Hkv > 0 && Hq == G * Hkv && window >= 1 && window <= 128;
}

size_t backward_tc_workspace_bytes(int B, int L, int Hq, int Hkv) {
    const size_t rq = static_cast<size_t>(B) * L * Hq, rk = static_cast<size_t>(B) * L * Hkv;
    return rq * D * 2 * 2 + rk * D * 2 + rq * 16;  // q_hat, dA, k_hat (bf16), statistics
}

cudaError_t launch_backward_tc(const BackwardTcParams& p, cudaStream_t s) {
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    if (nq == 0) return cudaSuccess;
    bwd_tc_prep_kernel<<<static_cast<unsigned>((nq + nk + 7) / 8), 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_qpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QP_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_kpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KP_SMEM);
    if (e != cudaSuccess) return e;
    const long long nbg = static_cast<long long>(p.B) * p.Hkv;
    bwd_qpass_kernel<<<static_cast<unsigned>(nbg * ((p.L + T - 1) / T)), kThreads, QP_SMEM, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_kpass_kernel<<<static_cast<unsigned>(nbg * ((p.L + BK - 1) / BK)), kThreads, KP_SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
