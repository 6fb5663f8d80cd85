// swa_prefill.cu -- gated sliding-window GQA attention prefill on sm_103a.
//
// Computes, for every query token i and query head h (KV head g = h / (Hq/Hkv)):
//   q_hat = RoPE(RMSNorm(q)), k_hat likewise;
//   A = softmax_j( q_hat . k_hat_j / sqrt(d) ) v_j  over j in [max(0, i-W+1), i];
//   out = A * sigmoid(gate)
// ("ZGCM-1-7B 完全解説", gotosocial explainer, section "アーキテクチャ":
// GatedSWA(h) = o_proj(A_SWA(q,k,v) ⊙ σ(g_proj(h))) over the most recent 128
// tokens; "ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for
// Math and Agentic Search", jaehun.me review, section "게이트형 SWA의 동작": the
// window counts the token itself, the gate multiplies element-wise.)
//
// Tiling.  One CTA owns one tile: T = 128/G consecutive tokens x the G query
// heads that share KV head g (GQA packing), i.e. an M = 128-row Q tile.  Its
// keys are the NK = T + 127 (rounded up to 16) tokens j0 = i0-127 .. i0+T-1,
// one K/V tile.  Four warps; thread t owns tile row t (TMEM lane t).
//   1. TMA: Q tile and K tile (128-byte swizzle) on one barrier, V on another.
//   2. every thread normalises + rotates its Q row and its K row(s) in smem
//      (bf16 in, fp16 out: the normalised values are bounded, see zg_qk.cuh).
//   3. one thread issues S = Q K^T (tcgen05, M128 x N=NK, fp32 in TMEM).
//   4. gate tile is fetched by TMA into the now-free Q buffer.
//   5. each thread reads its S row, masks it to the window, takes the exact
//      softmax (max, exp2, sum of the bf16-rounded weights) and writes P (bf16)
//      into the now-free K buffer in the K-major UMMA layout.
//   6. one thread issues O = P V (tcgen05, V read MN-major), into TMEM.
//   7. each thread scales its O row by 1/l and sigmoid(gate), writes bf16 into
//      the gate buffer in place; one thread TMA-stores the tile.
// Two CTAs fit per SM (112 KB smem, 256 TMEM columns each), so one CTA's
// memory phase overlaps the other's compute.
#include "zg_qk.cuh"

namespace zg {
namespace {

template <int D, int G>
struct SwaCfg {
    static constexpr int M = 128;                        // tile rows = G heads x T tokens
    static constexpr int T = M / G;                      // tokens per tile
    static constexpr int NK = ((T + 127) + 31) / 32 * 32;  // keys per tile (multiple of 32)
    static constexpr int NCH = D / 64;                   // 64-element chunks per head row
    static constexpr uint32_t Q_CHUNK = M * 128;         // bytes of one chunk of the Q tile
    static constexpr uint32_t K_CHUNK = NK * 128;
    static constexpr uint32_t Q_BYTES = Q_CHUNK * NCH;
    static constexpr uint32_t KV_BYTES = K_CHUNK * NCH;
    // P: K-major over keys; full 64-key chunks with 128-byte swizzle, a 32-key tail with 64-byte swizzle
    static constexpr int P_FULL = NK / 64;
    static constexpr int P_TAIL = NK % 64;  // 0 or 32 (NK is a multiple of 32)
    static constexpr uint32_t P_BYTES = P_FULL * (M * 128) + (P_TAIL ? M * 64 : 0);
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t KP_BYTES = (KV_BYTES > P_BYTES ? KV_BYTES : P_BYTES);
    static constexpr uint32_t OFF_V = ((OFF_K + KP_BYTES) + 1023) / 1024 * 1024;
    static constexpr uint32_t OFF_BAR = OFF_V + KV_BYTES;
    static constexpr uint32_t SMEM = OFF_BAR + 64;
    static constexpr uint32_t TMEM_COLS = 256;
    static_assert(NK <= 256 && NK % 32 == 0, "key tile");
    static_assert(P_TAIL == 0 || P_TAIL == 32, "P tail must be one 64-byte-swizzled chunk");
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(NK <= (int)TMEM_COLS && D <= (int)TMEM_COLS, "TMEM");
};

// PRE: inputs pre-normalised (q_hat, k_hat fp16; gate = sigmoid(g) bf16): transforms and sigmoid skipped
template <int D, int G, bool PRE>
__global__ void __launch_bounds__(128, 2) swa_prefill_kernel(const __grid_constant__ PrefillParams p) {
    using C = SwaCfg<D, G>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* bar_qk = bars + 0;
    uint64_t* bar_v = bars + 1;
    uint64_t* bar_g = bars + 2;
    uint64_t* bar_mma = bars + 3;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
    int* sflag = reinterpret_cast<int*>(bars + 5);

    const int t = threadIdx.x;
    const int warp = t >> 5;
    const int tile = blockIdx.x;
    const int lt = tile % p.n_ltiles;
    const int g = (tile / p.n_ltiles) % p.Hkv;
    const int b = tile / (p.n_ltiles * p.Hkv);
    const int i0 = lt * C::T;
    const int j0 = i0 - 127;  // first key of the tile (may be negative: zero-filled)

    if (t == 0) {
        *sflag = (smem_u32(smem) & 1023u) == 0 ? 1 : 0;
        if (!*sflag) report(p.ctl, 10, kErrAlign);
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_g, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = *sflag != 0;

    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    if (t == 0 && ok) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        mbar_arrive_expect_tx(bar_qk, C::Q_BYTES + C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
            tma_load_4d(sQ + c * C::Q_CHUNK, &p.tm_q, bar_qk, c * 64, g * G, i0, b);
            tma_load_4d(sK + c * C::K_CHUNK, &p.tm_k, bar_qk, c * 64, g, j0, b);
        }
        mbar_arrive_expect_tx(bar_v, C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) tma_load_4d(sV + c * C::K_CHUNK, &p.tm_v, bar_v, c * 64, g, j0, b);
    }

    // positions of this thread's rows (fetched while the tiles are in flight)
    const int tt = t / G;  // token of tile row t
    const int iq = i0 + tt;
    const int64_t seq = static_cast<int64_t>(b) * p.L;
    const int pos_q = iq < p.L && idx_ok(p.ctl, seq + iq, static_cast<long long>(p.B) * p.L, 86) ? __ldg(p.pos + seq + iq) : 0;
    int pos_k[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int kr = t + s * 128;
        const int j = j0 + kr;
        pos_k[s] = (kr < C::NK && j >= 0 && j < p.L && idx_ok(p.ctl, seq + j, static_cast<long long>(p.B) * p.L, 87))
                       ? __ldg(p.pos + seq + j)
                       : 0;
    }

    // ---- 2. QK-norm + RoPE in place
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_qk, 0, p.ctl, 11));
    if (ok && !PRE) {
        qk_norm_rope_row<D>(sQ, C::Q_CHUNK, t, p.wq, p.eps, pos_q, p.rope);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int kr = t + s * 128;
            if (kr < C::NK) qk_norm_rope_row<D>(sK, C::K_CHUNK, kr, p.wk, p.eps, pos_k[s], p.rope);
        }
    }
    if (!ok) *sflag = 0;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 3. S = Q K^T
    const uint32_t s_base = smem_u32(smem);
    if (t == 0 && *sflag) {
        constexpr uint32_t idesc = idesc_f16_f32(128, C::NK, false, false);  // q_hat, k_hat in fp16
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff = (ks & 3) * 32;
            const uint64_t a = sdesc(s_base + C::OFF_Q + (ks >> 2) * C::Q_CHUNK + koff, 16, 1024, kSw128);
            const uint64_t bdesc = sdesc(s_base + C::OFF_K + (ks >> 2) * C::K_CHUNK + koff, 16, 1024, kSw128);
            umma_bf16(tbase, a, bdesc, idesc, ks > 0);
        }
        umma_commit(bar_mma);
    }
    __syncthreads();
    ok = *sflag != 0;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 0, p.ctl, 12));
    tc_fence_after();
    __syncthreads();
    if (!ok) *sflag = 0;
    __syncthreads();
    ok = *sflag != 0;

    // ---- 4. gate tile into the Q buffer (Q has been consumed)
    if (t == 0 && ok) {
        mbar_arrive_expect_tx(bar_g, C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) tma_load_4d(sQ + c * C::Q_CHUNK, &p.tm_gate, bar_g, c * 64, g * G, i0, b);
    }

    // ---- 5. windowed softmax of row t -> P (bf16) in the K buffer
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(warp * 32) << 16);
    // valid key columns kr: j = j0 + kr in [max(0, iq - W + 1), iq]
    const int kr_lo = max(-j0, tt + 128 - p.window);
    const int kr_hi = tt + 127;
    float l_sum = 0.f;
    if (ok) {
        float m = -INFINITY;
#pragma unroll 1
        for (int cb = 0; cb < C::NK; cb += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int kr = cb + k;
                const float s = __uint_as_float(r[k]);
                if (kr >= kr_lo && kr <= kr_hi) m = fmaxf(m, s);
            }
        }
        const float mb = (m == -INFINITY ? 0.f : m) * p.scale_log2;
#pragma unroll 1
        for (int cb = 0; cb < C::NK; cb += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + cb, r);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const int kr = cb + k;
                float p0 = (kr >= kr_lo && kr <= kr_hi) ? ex2_approx(fmaf(__uint_as_float(r[k]), p.scale_log2, -mb)) : 0.f;
                float p1 = (kr + 1 >= kr_lo && kr + 1 <= kr_hi)
                               ? ex2_approx(fmaf(__uint_as_float(r[k + 1]), p.scale_log2, -mb))
                               : 0.f;
                pk[k / 2] = pack_bf16x2(p0, p1);
                l_sum += bf16lo(pk[k / 2]) + bf16hi(pk[k / 2]);
            }
            // 4 x 16-byte chunks of 8 keys
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int c8 = cb / 8 + q4;  // chunk of 8 keys, 0 .. NK/8-1
                if (c8 * 8 >= C::NK) break;
                uint32_t off;
                if (c8 < C::P_FULL * 8)
                    off = (c8 >> 3) * (128 * 128) + sw128_off(t, c8 & 7);
                else
                    off = C::P_FULL * (128 * 128) + sw64_off(t, c8 - C::P_FULL * 8);
                *reinterpret_cast<uint4*>(sK + off) =
                    make_uint4(pk[q4 * 4 + 0], pk[q4 * 4 + 1], pk[q4 * 4 + 2], pk[q4 * 4 + 3]);
            }
        }
    }
    if (!ok) *sflag = 0;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 6. O = P V
    if (t == 0 && *sflag) {
        bool vok = mbar_wait(bar_v, 0, p.ctl, 13);
        tc_fence_after();
        if (vok) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, D, false, true);
#pragma unroll
            for (int ks = 0; ks < C::NK / 16; ++ks) {
                uint64_t a;
                if (ks < C::P_FULL * 4)
                    a = sdesc(s_base + C::OFF_K + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024, kSw128);
                else
                    a = sdesc(s_base + C::OFF_K + C::P_FULL * (128 * 128) + (ks - C::P_FULL * 4) * 32, 16, 512, kSw64);
                // V tile: keys are rows (K dim), d contiguous (N dim, MN-major)
                const uint64_t bdesc = sdesc(s_base + C::OFF_V + ks * 16 * 128, C::K_CHUNK, 1024, kSw128);
                umma_bf16(tbase, a, bdesc, idesc, ks > 0);
            }
            umma_commit(bar_mma);
        } else {
            *sflag = 0;
        }
    }
    __syncthreads();
    ok = *sflag != 0;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma, 1, p.ctl, 14));
    tc_fence_after();
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar_g, 0, p.ctl, 15));

    // ---- 7. epilogue: out = O / l * sigmoid(gate), in place over the gate tile
    if (ok) {
        const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 32) {
            uint32_t r[32];
            tmem_ld32(lane_addr + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int e0 = cb + q4 * 8;
                uint8_t* gp = sQ + (e0 >> 6) * C::Q_CHUNK + sw128_off(t, (e0 & 63) >> 3);
                uint4 gv = *reinterpret_cast<const uint4*>(gp);
                const uint32_t gu[4] = {gv.x, gv.y, gv.z, gv.w};
                uint32_t ou[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float s0 = PRE ? bf16lo(gu[k]) : sigmoid_f32(bf16lo(gu[k]));
                    const float s1 = PRE ? bf16hi(gu[k]) : sigmoid_f32(bf16hi(gu[k]));
                    const float o0 = __uint_as_float(r[q4 * 8 + 2 * k]) * inv_l * s0;
                    const float o1 = __uint_as_float(r[q4 * 8 + 2 * k + 1]) * inv_l * s1;
                    ou[k] = pack_bf16x2(o0, o1);
                }
                *reinterpret_cast<uint4*>(gp) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
            }
        }
    }
    if (!ok) *sflag = 0;
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (t == 0 && *sflag) {
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) tma_store_4d(&p.tm_out, sQ + c * C::Q_CHUNK, c * 64, g * G, i0, b);
        bulk_commit();
        bulk_wait_read_all();
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, C::TMEM_COLS);
}

template <int D, int G>
cudaError_t launch_swa_t(const PrefillParams& p, cudaStream_t s) {
    using C = SwaCfg<D, G>;
    auto k = p.pre ? swa_prefill_kernel<D, G, true> : swa_prefill_kernel<D, G, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const long long tiles = static_cast<long long>(p.B) * p.Hkv * p.n_ltiles;
    k<<<static_cast<unsigned>(tiles), 128, C::SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int swa_kv_box_rows(int G) {
    const int T = 128 / G;
    if (swa2_supports(128, G)) return T;  // persistent kernel: one key slot of T tokens per copy
    return ((T + 127) + 31) / 32 * 32;    // one-tile kernel: the tile's whole key window
}

cudaError_t launch_swa_prefill(const PrefillParams& p, int d, cudaStream_t s) {
    const int G = p.Hq / p.Hkv;
    if (swa2_supports(d, G)) return launch_swa2_prefill(p, d, s);
    if (d == 128 && G == 4) return launch_swa_t<128, 4>(p, s);
    if (d == 64 && G == 4) return launch_swa_t<64, 4>(p, s);
    if (d == 128 && G == 8) return launch_swa_t<128, 8>(p, s);
    if (d == 64 && G == 8) return launch_swa_t<64, 8>(p, s);
    if (d == 128 && G == 2) return launch_swa_t<128, 2>(p, s);
    if (d == 64 && G == 2) return launch_swa_t<64, 2>(p, s);
    if (d == 128 && G == 1) return launch_swa_t<128, 1>(p, s);
    if (d == 64 && G == 1) return launch_swa_t<64, 1>(p, s);
    if (d == 128 && G == 16) return launch_swa_t<128, 16>(p, s);
    if (d == 64 && G == 16) return launch_swa_t<64, 16>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace zg
