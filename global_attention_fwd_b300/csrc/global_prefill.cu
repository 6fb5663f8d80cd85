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
// Kernel 2: one CTA per 128-row GQA tile (32 tokens x 4 heads of one KV
// head), heaviest tiles first.  Keys are consumed in blocks of 128:
//   S(kb) = Q K^T (fp16 tcgen05, TMEM, double-buffered so QK(kb+1) runs during
//   the softmax of block kb); each thread owns one row: online softmax with the
//   running max raised only when a block maximum exceeds it by 8 (log2 units),
//   then the O accumulator in TMEM is rescaled in place (rare); P (bf16) goes
//   to shared memory and O += P V (bf16 tcgen05, V read MN-major).
//   K_hat and V blocks arrive by TMA on separate two-stage rings: a K_hat stage
//   is refilled as soon as its QK has completed, a V stage after its PV.
// Only the last block of a tile can contain keys beyond the diagonal.
#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int D = 128;
constexpr int G = 4;
constexpr int T = 32;     // tokens per Q tile
constexpr int BK = 128;   // keys per block
constexpr uint32_t TILE = 128 * 128 * 2;  // one 128 x 128 16-bit tile (two 64-column chunks)
constexpr uint32_t CH = 128 * 128;        // bytes of one 64-column chunk of 128 rows
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + TILE;      // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE;  // 2 stages
constexpr uint32_t OFF_P = OFF_V + 2 * TILE;
constexpr uint32_t OFF_BAR = OFF_P + TILE;
constexpr uint32_t SMEM = OFF_BAR + 128;
constexpr uint32_t TMEM_COLS = 512;  // S0 [0,128), S1 [128,256), O [256,384)
constexpr float kTau = 8.0f;

// ---------------------------------------------------------------- kernel 1
__global__ void __launch_bounds__(256) khat_kernel(const __grid_constant__ PrefillParams p) {
    __shared__ float buf[8][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;  // (b, j, g) flattened
    const long long nrows = static_cast<long long>(p.B) * p.L * p.Hkv;
    if (row >= nrows) return;
    const long long tok = row / p.Hkv;  // b * L + j
    const int pos = __ldg(p.pos + tok);
    norm_rope_warp(p.k_raw + row * D, p.wk, p.eps, pos, p.rope, 1.0f, buf[warp]);
    const float4 v = *reinterpret_cast<const float4*>(&buf[warp][lane * 4]);
    uint2 o;
    o.x = pack_half2(v.x, v.y);
    o.y = pack_half2(v.z, v.w);
    *reinterpret_cast<uint2*>(p.khat + row * D + lane * 4) = o;
}

// ---------------------------------------------------------------- kernel 2
__global__ void __launch_bounds__(128, 1) global_attn_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* bar_q = bars + 0;
    uint64_t* bar_k = bars + 1;   // [2]
    uint64_t* bar_v = bars + 3;   // [2]
    uint64_t* bar_s = bars + 5;   // [2]
    uint64_t* bar_pv = bars + 7;
    uint64_t* bar_drain = bars + 8;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 9);
    int* sflag = reinterpret_cast<int*>(bars + 10);

    const int t = threadIdx.x, warp = t >> 5;
    // heaviest tiles (longest key ranges) first
    const int n_lt = p.n_ltiles;
    const int nbg = p.B * p.Hkv;
    const int lt = n_lt - 1 - static_cast<int>(blockIdx.x / nbg);
    const int g = static_cast<int>(blockIdx.x % nbg) % p.Hkv;
    const int b = static_cast<int>(blockIdx.x % nbg) / p.Hkv;
    const int i0 = lt * T;
    const int nkb = (i0 + T + BK - 1) / BK;

    uint8_t* sQ = smem + OFF_Q;
    uint8_t* sP = smem + OFF_P;
    if (t == 0) {
        *sflag = (smem_u32(smem) & 1023u) == 0 ? 1 : 0;
        if (!*sflag) report(p.ctl, 20, kErrAlign);
        mbar_init(bar_q, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_k[i], 1);
            mbar_init(&bar_v[i], 1);
            mbar_init(&bar_s[i], 1);
        }
        mbar_init(bar_pv, 1);
        mbar_init(bar_drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t sbase = smem_u32(smem);
    bool ok = *sflag != 0;

    auto load_k = [&](int kb) {
        uint64_t* bar = &bar_k[kb & 1];
        uint8_t* dst = smem + OFF_K + (kb & 1) * TILE;
        mbar_arrive_expect_tx(bar, TILE);
        tma_load_4d(dst, &p.tm_kh, bar, 0, g, kb * BK, b);
        tma_load_4d(dst + CH, &p.tm_kh, bar, 64, g, kb * BK, b);
    };
    auto load_v = [&](int kb) {
        uint64_t* bar = &bar_v[kb & 1];
        uint8_t* dst = smem + OFF_V + (kb & 1) * TILE;
        mbar_arrive_expect_tx(bar, TILE);
        tma_load_4d(dst, &p.tm_v, bar, 0, g, kb * BK, b);
        tma_load_4d(dst + CH, &p.tm_v, bar, 64, g, kb * BK, b);
    };
    auto issue_qk = [&](int kb) {
        constexpr uint32_t idesc = idesc_f16_f32(128, BK, false, false);
        const uint32_t kofs = OFF_K + (kb & 1) * TILE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t co = (ks >> 2) * CH + (ks & 3) * 32;
            umma_bf16(tbase + (kb & 1) * 128, sdesc(sbase + OFF_Q + co, 16, 1024, kSw128),
                      sdesc(sbase + kofs + co, 16, 1024, kSw128), idesc, ks > 0);
        }
        umma_commit(&bar_s[kb & 1]);
    };

    if (t == 0 && ok) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_kh);
        tma_prefetch_desc(&p.tm_v);
        mbar_arrive_expect_tx(bar_q, TILE);
        tma_load_4d(sQ, &p.tm_q, bar_q, 0, g * G, i0, b);
        tma_load_4d(sQ + CH, &p.tm_q, bar_q, 64, g * G, i0, b);
        load_k(0);
        load_v(0);
        if (nkb > 1) {
            load_k(1);
            load_v(1);
        }
    }
    const int tt = t / G;
    const int iq = i0 + tt;
    const int pos_q = iq < p.L ? __ldg(p.pos + static_cast<long long>(b) * p.L + iq) : 0;
    if (ok) ok = mbar_wait(bar_q, 0, p.ctl, 21);
    if (ok) qk_norm_rope_row<D>(sQ, CH, t, p.wq, p.eps, pos_q, p.rope);
    if (!ok) *sflag = 0;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t == 0 && *sflag) {
        if (mbar_wait(&bar_k[0], 0, p.ctl, 22)) {
            tc_fence_after();
            issue_qk(0);
        } else {
            *sflag = 0;
        }
    }
    __syncthreads();
    ok = *sflag != 0;

    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t o_col = 256;
    float m_run = -INFINITY, l_run = 0.f;
    for (int kb = 0; kb < nkb; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_s[kb & 1], (kb >> 1) & 1, p.ctl, 23));
        tc_fence_after();
        if (t == 0 && ok) {
            if (kb + 2 < nkb) load_k(kb + 2);  // K stage kb&1 is free: QK(kb) has completed
            if (kb + 1 < nkb) {
                if (mbar_wait(&bar_k[(kb + 1) & 1], ((kb + 1) >> 1) & 1, p.ctl, 24))
                    issue_qk(kb + 1);
                else
                    *sflag = 0;
            }
        }
        // ---- row max of block kb
        const bool last = kb == nkb - 1;
        if (!ok) *sflag = 0;
        const int kmax = iq - kb * BK;  // last valid key column of this row in the block
        const uint32_t s_addr = lane_addr + (kb & 1) * 128;
        float mb = -INFINITY;
#pragma unroll 1
        for (int cb = 0; cb < BK && ok; cb += 32) {
            uint32_t r[32];
            tmem_ld32(s_addr + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (!last || cb + k <= kmax) mb = fmaxf(mb, __uint_as_float(r[k]));
        }
        mb *= p.scale_log2;
        float m_new = m_run;
        if (mb > m_run + kTau || m_run == -INFINITY) m_new = mb;
        const float corr = m_run == -INFINITY ? 0.f : ex2_approx(m_run - m_new);
        // ---- previous PV must be done: P buffer free, O stable, V stage (kb-1)&1 free
        if (kb > 0) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bar_pv, (kb - 1) & 1, p.ctl, 25));
            tc_fence_after();
            if (t == 0 && ok && kb + 1 < nkb) load_v(kb + 1);
            // rescale O where the running max moved (warp-uniform TMEM access)
            if (ok && __any_sync(0xffffffffu, m_new != m_run)) {
#pragma unroll 1
                for (int cb = 0; cb < D; cb += 32) {
                    uint32_t r[32];
                    tmem_ld32(lane_addr + o_col + cb, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * corr);
                    tmem_st32(lane_addr + o_col + cb, r);
                }
                tmem_wait_st();
            }
        }
        l_run *= corr;
        m_run = m_new;
        // ---- P = exp2(S * scale - m) in bf16 -> shared memory (K-major, 128-byte swizzle)
#pragma unroll 1
        for (int cb = 0; cb < BK && ok; cb += 32) {
            uint32_t r[32];
            tmem_ld32(s_addr + cb, r);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const float p0 = (!last || cb + k <= kmax) ? ex2_approx(fmaf(__uint_as_float(r[k]), p.scale_log2, -m_run)) : 0.f;
                const float p1 =
                    (!last || cb + k + 1 <= kmax) ? ex2_approx(fmaf(__uint_as_float(r[k + 1]), p.scale_log2, -m_run)) : 0.f;
                pk[k / 2] = pack_bf16x2(p0, p1);
                l_run += bf16lo(pk[k / 2]) + bf16hi(pk[k / 2]);
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int c8 = cb / 8 + q4;
                *reinterpret_cast<uint4*>(sP + (c8 >> 3) * CH + sw128_off(t, c8 & 7)) =
                    make_uint4(pk[q4 * 4], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
            }
        }
        if (!ok) *sflag = 0;
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        ok = *sflag != 0;
        if (!ok) break;  // uniform: every thread read the same flag after the barrier
        if (t == 0 && ok) {
            if (mbar_wait(&bar_v[kb & 1], (kb >> 1) & 1, p.ctl, 26)) {
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16_f32(128, D, false, true);
                const uint32_t vofs = OFF_V + (kb & 1) * TILE;
#pragma unroll
                for (int ks = 0; ks < BK / 16; ++ks) {
                    const uint64_t a = sdesc(sbase + OFF_P + (ks >> 2) * CH + (ks & 3) * 32, 16, 1024, kSw128);
                    const uint64_t bd = sdesc(sbase + vofs + ks * 16 * 128, CH, 1024, kSw128);
                    umma_bf16(tbase + o_col, a, bd, idesc, (kb > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(bar_pv);
            } else {
                *sflag = 0;
            }
        }
    }
    // ---- epilogue: O / l -> bf16 -> shared memory (Q buffer) -> TMA store
    __syncthreads();
    ok = *sflag != 0;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_pv, (nkb - 1) & 1, p.ctl, 27));
    tc_fence_after();
    if (ok) {
        const float inv_l = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + o_col + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t ou[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ou[k] = pack_bf16x2(__uint_as_float(r[q4 * 8 + 2 * k]) * inv_l,
                                        __uint_as_float(r[q4 * 8 + 2 * k + 1]) * inv_l);
                const int e0 = cb + q4 * 8;
                *reinterpret_cast<uint4*>(sQ + (e0 >> 6) * CH + sw128_off(t, (e0 & 63) >> 3)) =
                    make_uint4(ou[0], ou[1], ou[2], ou[3]);
            }
        }
    }
    if (!ok) *sflag = 0;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0 && *sflag) {
        tma_store_4d(&p.tm_out, sQ, 0, g * G, i0, b);
        tma_store_4d(&p.tm_out, sQ + CH, 64, g * G, i0, b);
        bulk_commit();
        bulk_wait_read_all();
    }
    if (t == 0 && !*sflag) {
        // abandoned tile: wait (bounded) for every MMA this thread issued, then give
        // copies still in flight a millisecond to land before the CTA releases its memory
        umma_commit(bar_drain);
        (void)mbar_wait(bar_drain, 0, p.ctl, 28);
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, TMEM_COLS);
}

}  // namespace

int global_q_tile_tokens() { return T; }

cudaError_t launch_global_prefill(const PrefillParams& p, int d, cudaStream_t s) {
    if (d != D || p.Hq != p.Hkv * G) return cudaErrorInvalidValue;
    const long long rows = static_cast<long long>(p.B) * p.L * p.Hkv;
    khat_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(global_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.B) * p.Hkv * p.n_ltiles;
    global_attn_kernel<<<static_cast<unsigned>(ctas), 128, SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
