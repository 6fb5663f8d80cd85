// hybrid_decode.cu -- one decode step through the hybrid layer stack.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ": 27 local
// layers keep a KV cache of the last 128 tokens, the 5 global layers keep the
// whole sequence; decode is bound by memory bandwidth, so its cost is the cache
// it reads.  "ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for
// Math and Agentic Search" (jaehun.me review), section "KV 캐시가 6.4배 줄어드는
// 이유": 20 KiB of cache per token (5 global layers x 8 KV heads x 128 x K,V x
// bf16).
//
// Per layer l, sequence b, KV head g (G = Hq / Hkv query heads), new token at p:
//   q_hat, k_hat = RoPE(RMSNorm(.)) at p; k_hat and v_new go to the cache
//   (global layer: slot p; local layer: ring slot p mod W); the G query heads
//   attend to positions 0..p (global) or max(0, p-W+1)..p (local, gated).
//
// Kernel 1 (attention, split-K).  One CTA per (global layer, b, g, split of
// 8192 keys) and per (local layer, b, g); two CTAs per SM.  Warp 3 streams the
// cache slice into a ring of three stages in shared memory with 2-D TMA copies
// (16 KB of K and 16 KB of V per stage, 128-byte swizzle, so the fragment loads
// below are free of bank conflicts).  Warps 0-2 each own one stage buffer and
// take every third stage.  For one GQA group the scores are a small dense
// product (G <= 16 query rows), so each warp runs it on the warp-level tensor
// core instruction (mma.sync m16n8k16, fp32 accumulate) with the G heads as the
// 16 rows: S = Q_hat K^T (Q_hat split into a bf16 head and a bf16 tail, so the
// scores keep ~16 mantissa bits), an online softmax on the accumulator
// fragments (max raised only when a score exceeds it by 8 in log2 units), then
// O^T = V^T P^T with P taken straight from the score fragments.  That costs a
// few instructions per key instead of a per-key chain of shuffle reductions, so
// the stream runs at HBM rate.  The partials of the three warps and of the new
// key (added in fp32) are merged in shared memory; global splits write (m, l, o)
// to the workspace, local layers finish in place (1/l, sigmoid gate, bf16).  The
// CTA that owns position p also writes the new cache slot.
// Kernel 2 merges the splits of every global (layer, b, head) in a fixed order.
//
// FP8 caches use E4M3, the forward FP8 format of the training recipe in
// "ZGCM-1-7B 完全解説", section "学習の高速化 — FP8・Muon・TWEOが生む約4.2倍の効率".
// They hold e4m3(k_hat * k_scale) and e4m3(v * v_scale): a stage carries twice
// the keys; fragments are loaded as bytes and widened to fp16 in registers
// (exactly), and the products run in fp16 with fp32 accumulation.  1 / k_scale
// is folded into q_hat, 1 / v_scale into the output.  RMSNorm bounds |k_hat| by
// sqrt(d) max|wk|, far inside the E4M3 range.
#include <cuda_fp8.h>

#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int NCW = 3;               // consumer warps; warp w owns stage buffer w
constexpr int NST = NCW;             // stages in the ring
constexpr int NTHR = (NCW + 1) * 32;
constexpr uint32_t STAGE_T = 16384;  // bytes of K (and of V) per stage
constexpr int KSUB = 64;             // keys per softmax sub-block (8 n-tiles of 8 keys)
constexpr float kLazy = 8.0f;        // raise the running max only past this margin (log2 units)

template <int D, bool FP8>
struct Dec {
    static constexpr int EB = FP8 ? 1 : 2;                   // bytes per cache element
    static constexpr int ROWB = D * EB;                      // bytes per cache row
    static constexpr int KPS = STAGE_T / ROWB;               // keys per stage
    static constexpr int RB = ROWB < 128 ? ROWB : 128;       // bytes per swizzled smem row (one TMA box row)
    static constexpr int NCHK = ROWB / RB;                   // TMA boxes per stage and tensor
    static constexpr int UPR = RB / 16;                      // 16-byte units per smem row
    static constexpr int NMT = D / 16;                       // 16-dim tiles of O^T
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = NST * STAGE_T;
    static constexpr uint32_t OFF_QH = 2 * NST * STAGE_T;    // q_hat [16][D] f32 (x scale_log2 / k_scale)
    static constexpr uint32_t OFF_KH = OFF_QH + 16 * D * 4;  // k_hat [D] f32
    static constexpr uint32_t OFF_VN = OFF_KH + D * 4;       // v_new [D] f32
    static constexpr uint32_t OFF_RED = OFF_VN + D * 4;      // (m, l) of the NCW + 1 partials x 16 heads
    static constexpr uint32_t OFF_BAR = OFF_RED + (NCW + 1) * 16 * 2 * 4;
    static constexpr uint32_t SMEM = OFF_BAR + 64;
    static_assert(KPS % KSUB == 0 && KPS <= 256, "stage shape");
    static_assert(RB == 128 || RB == 64, "swizzle width");
    static_assert((NCW + 1) * 16 * D * 4 <= 2 * NST * STAGE_T, "partials fit in the stage area");
    static_assert(2 * (SMEM + 1024) <= 232448, "two CTAs per SM");
};

// byte offset of 16-byte unit u (0 .. ROWB/16-1) of row r in a stage written by TMA with
// RB-byte box rows (128- or 64-byte swizzle), NCHK boxes of KPS rows one after the other
template <int D, bool FP8>
__device__ __forceinline__ uint32_t sw_addr(uint32_t r, uint32_t u) {
    using C = Dec<D, FP8>;
    const uint32_t ch = u / C::UPR, uu = u % C::UPR;
    const uint32_t swz = C::RB == 128 ? (r & 7u) : ((r >> 1) & 3u);
    return ch * (C::KPS * C::RB) + r * C::RB + ((uu ^ swz) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// C (16x8, fp32) += A (16x16) B (16x8); bf16 or fp16 operands
template <bool F16>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    if (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// four E4M3 values (low byte first) -> two fp16 pairs (bytes 0,1 and bytes 2,3), exactly
__device__ __forceinline__ void e4m3x4_to_h2(uint32_t x, uint32_t& lo, uint32_t& hi) {
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b; }"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ float h2sum(uint32_t u) {
    const __half2 h = *reinterpret_cast<const __half2*>(&u);
    return __low2float(h) + __high2float(h);
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

template <int D, bool FP8, int NH>
__global__ void __launch_bounds__(NTHR, 2) decode_attn_kernel(const __grid_constant__ DecodeParams p) {
    using C = Dec<D, FP8>;
    constexpr int KPS = C::KPS;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + NST;
    int* sflag = reinterpret_cast<int*>(empty + NST);
    float* qh = reinterpret_cast<float*>(smem + C::OFF_QH);
    float* kh = reinterpret_cast<float*>(smem + C::OFF_KH);
    float* vn = reinterpret_cast<float*>(smem + C::OFF_VN);
    float* red_ml = reinterpret_cast<float*>(smem + C::OFF_RED);  // [NCW + 1][16][2]
    float* red_o = reinterpret_cast<float*>(smem);                 // [NCW + 1][16][D], over the stages at the end

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.Hq / p.Hkv;
    // ---- which work item
    const long long n_glob = static_cast<long long>(p.NG) * p.B * p.Hkv * p.nsplit;
    const long long bid = blockIdx.x;
    const bool is_glob = bid < n_glob;
    int layer, lidx, b, g, split = 0;
    long long slice;  // (layer index, b, g): the outer coordinate of the cache tensor maps
    if (is_glob) {
        split = static_cast<int>(bid % p.nsplit);
        slice = bid / p.nsplit;
        layer = p.layer_of_global[slice / (static_cast<long long>(p.Hkv) * p.B)];
    } else {
        slice = bid - n_glob;
        layer = p.layer_of_local[slice / (static_cast<long long>(p.Hkv) * p.B)];
    }
    g = static_cast<int>(slice % p.Hkv);
    b = static_cast<int>((slice / p.Hkv) % p.B);
    lidx = static_cast<int>(slice / (static_cast<long long>(p.Hkv) * p.B));
    const int pos = idx_ok(p.ctl, b, p.B, 70) ? __ldg(p.pos + b) : -1;
    const bool pos_ok = pos >= 0 && static_cast<long long>(pos) < p.S;
    // the new token's cache row (debug builds check it before the slot is written)
    const long long slot_row = is_glob ? slice * p.S + pos : slice * p.W + (pos_ok ? pos % p.W : 0);
    const long long slot_rows = is_glob ? static_cast<long long>(p.NG) * p.B * p.Hkv * p.S
                                        : static_cast<long long>(p.NS) * p.B * p.Hkv * p.W;
    // keys streamed from the cache: [k0, k0 + nk) of the slice; whether this CTA owns p
    long long k0 = 0;
    int nk = 0;
    bool owner;
    uint8_t *kslot, *vslot;
    if (is_glob) {
        k0 = static_cast<long long>(split) * p.split_len;
        long long k1 = k0 + p.split_len;
        if (pos_ok && k1 > pos) k1 = pos;
        nk = pos_ok && k1 > k0 ? static_cast<int>(k1 - k0) : 0;
        owner = pos_ok && pos / p.split_len == split;
        const size_t row = static_cast<size_t>(slice) * static_cast<size_t>(p.S) + (pos_ok ? pos : 0);
        kslot = reinterpret_cast<uint8_t*>(p.k_glob) + row * C::ROWB;
        vslot = reinterpret_cast<uint8_t*>(p.v_glob) + row * C::ROWB;
    } else {
        nk = pos_ok ? p.W : 0;  // every slot is streamed; invalid ones are masked
        owner = pos_ok;
        const size_t row = static_cast<size_t>(slice) * p.W + (pos_ok ? pos % p.W : 0);
        kslot = reinterpret_cast<uint8_t*>(p.k_ring) + row * C::ROWB;
        vslot = reinterpret_cast<uint8_t*>(p.v_ring) + row * C::ROWB;
    }
    const int nstage = (nk + KPS - 1) / KPS;
    const CUtensorMap* mk = is_glob ? &p.tm_kg : &p.tm_kr;
    const CUtensorMap* mv = is_glob ? &p.tm_vg : &p.tm_vr;

    if (threadIdx.x == 0) {
        *sflag = (smem_u32(smem) & 1023u) == 0 ? 1 : 0;
        if (!*sflag) report(p.ctl, 45, kErrAlign);
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // one stage of K and V: rows [k0 + st * KPS, + KPS) of the slice (rows past the slice's
    // slots read as zeros); issued by one thread
    auto issue_stage = [&](int st) {
        const int bf = st % NST;
        mbar_arrive_expect_tx(&full[bf], 2u * STAGE_T);
        const int row = static_cast<int>(k0) + st * KPS;
#pragma unroll
        for (int ch = 0; ch < C::NCHK; ++ch) {
            tma_load_3d(smem + C::OFF_K + bf * STAGE_T + ch * (KPS * C::RB), mk, &full[bf], ch * (C::RB / C::EB), row,
                        static_cast<int>(slice));
            tma_load_3d(smem + C::OFF_V + bf * STAGE_T + ch * (KPS * C::RB), mv, &full[bf], ch * (C::RB / C::EB), row,
                        static_cast<int>(slice));
        }
    };

    if (warp == NCW) {
        // ---------------- producer (lane 0), the new key (whole warp)
        const int first = min(nstage, NST);
        if (lane == 0 && *sflag) {
            tma_prefetch_desc(mk);
            tma_prefetch_desc(mv);
            for (int st = 0; st < first; ++st) issue_stage(st);  // the ring starts empty: no waits
        }
        if (owner && *sflag && idx_ok(p.ctl, slot_row, slot_rows, 71) &&
            idx_ok(p.ctl, (static_cast<long long>(layer) * p.B + b) * p.Hkv + g,
                   static_cast<long long>(p.NL) * p.B * p.Hkv, 72)) {
            const size_t tok = static_cast<size_t>(layer) * p.B + b;
            norm_rope_warp_d<D>(p.k_new + (tok * p.Hkv + g) * D, p.wk + static_cast<size_t>(layer) * D, p.eps, pos,
                                p.rope, 1.0f, kh);
            const __nv_bfloat16* vx = p.v_new + (tok * p.Hkv + g) * D;
            for (int e = lane; e < D; e += 32) vn[e] = __bfloat162float(vx[e]);
            __syncwarp();
            // the new cache slot: normalised + rotated key, raw value
            if (FP8) {
                for (int e = 2 * lane; e < D; e += 64) {
                    *reinterpret_cast<__nv_fp8x2_storage_t*>(kslot + e) = __nv_cvt_float2_to_fp8x2(
                        make_float2(kh[e] * p.k_scale, kh[e + 1] * p.k_scale), __NV_SATFINITE, __NV_E4M3);
                    *reinterpret_cast<__nv_fp8x2_storage_t*>(vslot + e) = __nv_cvt_float2_to_fp8x2(
                        make_float2(vn[e] * p.v_scale, vn[e + 1] * p.v_scale), __NV_SATFINITE, __NV_E4M3);
                }
            } else {
                for (int e = lane; e < D; e += 32) {
                    reinterpret_cast<__nv_bfloat16*>(kslot)[e] = __float2bfloat16_rn(kh[e]);
                    reinterpret_cast<__nv_bfloat16*>(vslot)[e] = vx[e];
                }
            }
        }
        if (lane == 0 && *sflag) {
            bool ok = true;
            int issued = first;
            for (int st = first; st < nstage && ok; ++st) {
                ok = mbar_wait(&empty[st % NST], ((st / NST) - 1) & 1, p.ctl, 46);
                if (!ok) break;
                issue_stage(st);
                ++issued;
            }
            if (!ok) {
                *sflag = 0;
                // every issued copy must land before the CTA may exit
                for (int st = max(0, issued - NST); st < issued; ++st)
                    (void)mbar_wait(&full[st % NST], (st / NST) & 1, p.ctl, 47);
            }
        }
        __syncthreads();  // (1)
        // the new key's partial (owner only): m = its score, l = 1, o = v_new (in stored units)
        const float vs = FP8 ? p.v_scale : 1.0f;
        const float kscale = FP8 ? p.k_scale : 1.0f;  // q_hat carries 1 / k_scale
        for (int h = 0; h < G; ++h) {
            float sc = -INFINITY;
            if (owner && *sflag) {
                float acc = 0.f;
                for (int e = lane; e < D; e += 32) acc = fmaf(qh[h * D + e] * kscale, kh[e], acc);
#pragma unroll
                for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                sc = acc;
            }
            if (lane == 0) {
                red_ml[(NCW * 16 + h) * 2 + 0] = sc;
                red_ml[(NCW * 16 + h) * 2 + 1] = sc == -INFINITY ? 0.f : 1.f;
            }
            if (sc != -INFINITY)
                for (int e = lane; e < D; e += 32) red_o[(NCW * 16 + h) * D + e] = vn[e] * vs;
        }
    } else {
        // ---------------- consumers: q_hat of heads warp, warp + NCW, ...
        if (pos_ok) {
            const size_t tok = static_cast<size_t>(layer) * p.B + b;
            const float qscale = FP8 ? p.scale_log2 / p.k_scale : p.scale_log2;  // scores in log2 units
            for (int h = warp; h < G; h += NCW)
                if (idx_ok(p.ctl, static_cast<long long>(tok * p.Hq + static_cast<size_t>(g) * G + h),
                           static_cast<long long>(p.NL) * p.B * p.Hq, 73))
                    norm_rope_warp_d<D>(p.q + (tok * p.Hq + static_cast<size_t>(g) * G + h) * D,
                                    p.wq + static_cast<size_t>(layer) * D, p.eps, pos, p.rope, qscale, qh + h * D);
        }
        asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");

        const int gq = lane >> 2, tg = lane & 3;  // fragment row group, thread in the group
        // A fragments of Q_hat (16 rows = heads, zero past G), one per k-step of 16 dims.  bf16
        // caches: Q_hat = hi + lo, both bf16.  E4M3 caches: fp16, with the dims of each k-step
        // permuted to match the byte layout of the key fragments (see the product below).
        uint32_t qa[D / 16][4], ql[FP8 ? 1 : D / 16][4];
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int h = gq + (r & 1) * 8;
                const int e0 = FP8 ? 16 * ks + 4 * tg + (r >> 1) * 2   // dims 4tg, 4tg+1 | 4tg+2, 4tg+3
                                   : 16 * ks + 2 * tg + (r >> 1) * 8;  // dims 2tg, 2tg+1 | 2tg+8, 2tg+9
                const float x0 = h < G ? qh[h * D + e0] : 0.f, x1 = h < G ? qh[h * D + e0 + 1] : 0.f;
                if (FP8) {
                    qa[ks][r] = pack_half2(x0, x1);
                } else {
                    const uint32_t hi = pack_bf16x2(x0, x1);
                    qa[ks][r] = hi;
                    ql[FP8 ? 0 : ks][r] = pack_bf16x2(x0 - bf16lo(hi), x1 - bf16hi(hi));
                }
            }
        }
        float o[C::NMT][NH][4];
#pragma unroll
        for (int mt = 0; mt < C::NMT; ++mt)
#pragma unroll
            for (int hg = 0; hg < NH; ++hg)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[mt][hg][r] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // heads gq, gq + 8
        const bool ring = !is_glob;
        const int wslot = pos_ok ? pos % p.W : -1;
        auto key_ok = [&](int key) {  // key: index in the streamed slice
            if (key >= nk) return false;
            if (ring) return key != wslot && (pos >= p.W - 1 || key < pos);
            return true;
        };
        const int bf = warp;  // this warp's stage buffer
        const uint32_t kbase = smem_u32(smem + C::OFF_K + bf * STAGE_T);
        const uint32_t vbase = smem_u32(smem + C::OFF_V + bf * STAGE_T);
        bool ok = true;
        for (int st = warp; st < nstage; st += NCW) {
            ok = *sflag && mbar_wait(&full[bf], (st / NST) & 1, p.ctl, 48);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            bool wrote = false;
#pragma unroll 1
            for (int sb = 0; sb < KPS / KSUB; ++sb) {
                const int key0 = st * KPS + sb * KSUB;  // first key of the sub-block in the slice
                if (key0 >= nk) break;
                const bool edge = key0 + KSUB > nk || ring;  // the sub-block may hold keys to mask
                // ---- S = Q_hat K^T: 8 n-tiles of 8 keys, fp32 accumulators
                float s[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) s[nt][r] = 0.f;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const uint32_t row = sb * KSUB + nt * 8 + (lane & 7);
                    if (FP8) {
                        // one x4 = 8 keys x 64 byte-dims: register i holds dims 16i + 4tg .. +3 of key gq
#pragma unroll
                        for (int grp = 0; grp < D / 64; ++grp) {
                            uint32_t kr[4];
                            ldsm_x4(kbase + sw_addr<D, FP8>(row, 4 * grp + (lane >> 3)), kr);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int ks = 4 * grp + i;
                                uint32_t b0, b1;
                                e4m3x4_to_h2(kr[i], b0, b1);
                                mma16816<true>(s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                            }
                        }
                    } else {
                        // one x4 = 8 keys x 32 dims: registers (0, 1) and (2, 3) are two k-steps
#pragma unroll
                        for (int grp = 0; grp < D / 32; ++grp) {
                            uint32_t kr[4];
                            ldsm_x4(kbase + sw_addr<D, FP8>(row, 4 * grp + (lane >> 3)), kr);
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int ks = 2 * grp + i;
                                mma16816<false>(s[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kr[2 * i],
                                                kr[2 * i + 1]);
                                mma16816<false>(s[nt], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], kr[2 * i],
                                                kr[2 * i + 1]);
                            }
                        }
                    }
                }
                // ---- masking: scores by selection; V rows of masked keys zeroed (0 * NaN is NaN)
                if (edge) {
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            if (!key_ok(key0 + nt * 8 + 2 * tg + (r & 1))) s[nt][r] = -INFINITY;
                    constexpr int UPK = C::ROWB / 16;  // 16-byte units per key row
                    for (int idx = lane; idx < KSUB * UPK; idx += 32) {
                        const int kr = idx / UPK;
                        if (!key_ok(key0 + kr)) {
                            *reinterpret_cast<uint4*>(smem + C::OFF_V + bf * STAGE_T +
                                                      sw_addr<D, FP8>(sb * KSUB + kr, idx % UPK)) =
                                make_uint4(0u, 0u, 0u, 0u);
                            wrote = true;
                        }
                    }
                    __syncwarp();
                }
                // ---- online softmax on the fragments: rows gq (r = 0, 1) and gq + 8 (r = 2, 3)
                float corr[2] = {1.f, 1.f};
                bool raise = false;
#pragma unroll
                for (int hg = 0; hg < NH; ++hg) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * hg], s[nt][2 * hg + 1]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    if (mx != -INFINITY && (m_run[hg] == -INFINITY || mx > m_run[hg] + kLazy)) {
                        corr[hg] = m_run[hg] == -INFINITY ? 0.f : ex2_approx(m_run[hg] - mx);
                        m_run[hg] = mx;
                        l_run[hg] *= corr[hg];
                        raise = true;
                    }
                }
                if (__any_sync(0xffffffffu, raise)) {
                    // the O^T columns of this thread are heads 2tg, 2tg + 1 (+ 8 per head group)
#pragma unroll
                    for (int hg = 0; hg < NH; ++hg) {
                        const float c0 = __shfl_sync(0xffffffffu, corr[hg], (2 * tg) * 4);
                        const float c1 = __shfl_sync(0xffffffffu, corr[hg], (2 * tg + 1) * 4);
#pragma unroll
                        for (int mt = 0; mt < C::NMT; ++mt) {
                            o[mt][hg][0] *= c0;
                            o[mt][hg][1] *= c1;
                            o[mt][hg][2] *= c0;
                            o[mt][hg][3] *= c1;
                        }
                    }
                }
                // P = 2^(s - m), packed as the B operand of O^T = V^T P^T (k = keys, n = heads)
                uint32_t pb[NH][4][2];
#pragma unroll
                for (int hg = 0; hg < NH; ++hg) {
                    const float mu = m_run[hg] == -INFINITY ? 0.f : m_run[hg];
                    float ls = 0.f;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt) {
                        const float p0 = ex2_approx(s[nt][2 * hg] - mu), p1 = ex2_approx(s[nt][2 * hg + 1] - mu);
                        const uint32_t pk = FP8 ? pack_half2(p0, p1) : pack_bf16x2(p0, p1);
                        ls += FP8 ? h2sum(pk) : bf16lo(pk) + bf16hi(pk);  // sums of the very values used
                        pb[hg][nt >> 1][nt & 1] = pk;
                    }
                    l_run[hg] += ls;
                }
                // ---- O^T += V^T P^T per 16-dim tile and 16-key step
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t rbase = sb * KSUB + kk * 16;
                    const int i = lane >> 3;
                    if (FP8) {
                        // x4.trans on bytes: matrices (keys 0-7 | 8-15) x (dim block 2j | 2j+1); a register
                        // holds dims (2gq, 2gq+1) of keys 2tg, 2tg+1 -> tile rows gq (even dims), gq+8 (odd)
#pragma unroll
                        for (int j = 0; j < C::NMT / 2; ++j) {
                            uint32_t vr[4];
                            ldsm_x4_t(vbase + sw_addr<D, FP8>(rbase + (lane & 7) + 8 * (i & 1), 2 * j + (i >> 1)), vr);
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t x0, y0, x1, y1;
                                e4m3x4_to_h2(vr[2 * half], x0, y0);
                                e4m3x4_to_h2(vr[2 * half + 1], x1, y1);
                                const uint32_t a0 = prmt(x0, y0, 0x5410), a1 = prmt(x0, y0, 0x7632);
                                const uint32_t a2 = prmt(x1, y1, 0x5410), a3 = prmt(x1, y1, 0x7632);
#pragma unroll
                                for (int hg = 0; hg < NH; ++hg)
                                    mma16816<true>(o[2 * j + half][hg], a0, a1, a2, a3, pb[hg][kk][0], pb[hg][kk][1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int mt = 0; mt < C::NMT; ++mt) {
                            uint32_t vr[4];
                            ldsm_x4_t(vbase + sw_addr<D, FP8>(rbase + (lane & 7) + 8 * (i >> 1), 2 * mt + (i & 1)), vr);
#pragma unroll
                            for (int hg = 0; hg < NH; ++hg)
                                mma16816<false>(o[mt][hg], vr[0], vr[1], vr[2], vr[3], pb[hg][kk][0], pb[hg][kk][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (wrote) fence_async_smem();  // the zeroed rows before the next copy into the buffer
                mbar_arrive(&empty[bf]);
            }
        }
        if (!ok) *sflag = 0;
        // ---- this warp's partial; l summed over the four threads of a row group
#pragma unroll
        for (int hg = 0; hg < NH; ++hg) {
            l_run[hg] += __shfl_xor_sync(0xffffffffu, l_run[hg], 1);
            l_run[hg] += __shfl_xor_sync(0xffffffffu, l_run[hg], 2);
        }
        __syncthreads();  // (1) every warp is past the stages: the stage area takes the partials
#pragma unroll
        for (int hg = 0; hg < NH; ++hg) {
            if (tg == 0) {
                red_ml[(warp * 16 + gq + 8 * hg) * 2 + 0] = m_run[hg];
                red_ml[(warp * 16 + gq + 8 * hg) * 2 + 1] = l_run[hg];
            }
#pragma unroll
            for (int mt = 0; mt < C::NMT; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int h = 8 * hg + 2 * tg + (r & 1);
                    // tile row -> dim: bf16 tiles hold 16 consecutive dims; E4M3 tiles hold the even
                    // (rows 0-7) and the odd (rows 8-15) dims of a 16-dim block
                    const int dim = FP8 ? 16 * mt + 2 * gq + (r >> 1) : 16 * mt + gq + 8 * (r >> 1);
                    red_o[(warp * 16 + h) * D + dim] = o[mt][hg][r];
                }
        }
    }
    __syncthreads();  // (2) the partials are complete
    const bool all_ok = *sflag != 0;
    const float inv_vs = FP8 ? 1.0f / p.v_scale : 1.0f;
    for (int idx = threadIdx.x; idx < G * D; idx += NTHR) {
        const int h = idx / D, e = idx % D;
        float mt = -INFINITY;
#pragma unroll
        for (int w = 0; w <= NCW; ++w) mt = fmaxf(mt, red_ml[(w * 16 + h) * 2]);
        float lt = 0.f, ot = 0.f;
#pragma unroll
        for (int w = 0; w <= NCW; ++w) {
            const float mw = red_ml[(w * 16 + h) * 2];
            if (mw == -INFINITY) continue;
            const float c = ex2_approx(mw - mt);
            lt += red_ml[(w * 16 + h) * 2 + 1] * c;
            ot += red_o[(w * 16 + h) * D + e] * c;
        }
        ot *= inv_vs;
        const int hq = g * G + h;
        if (is_glob) {
            const size_t row = ((static_cast<size_t>(lidx) * p.B + b) * p.Hq + hq) * p.nsplit + split;
            if (!idx_ok(p.ctl, static_cast<long long>(row), static_cast<long long>(p.NG) * p.B * p.Hq * p.nsplit, 74))
                continue;
            p.ws_o[row * D + e] = (all_ok ? ot : 0.f);
            if (e == 0) {
                p.ws_ml[row * 2 + 0] = all_ok ? mt : -INFINITY;
                p.ws_ml[row * 2 + 1] = all_ok ? lt : 0.f;
            }
        } else {
            const size_t orow = (static_cast<size_t>(layer) * p.B + b) * p.Hq + hq;
            if (!idx_ok(p.ctl, static_cast<long long>(orow), static_cast<long long>(p.NL) * p.B * p.Hq, 75)) continue;
            float r = 0.f;
            if (all_ok && lt > 0.f) r = ot / lt * sigmoid_f32(__bfloat162float(p.gate[orow * D + e]));
            p.out[orow * D + e] = __float2bfloat16_rn(r);
        }
    }
}

// merge the splits of one (global layer, b, query head): D threads, one per dim
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
    const int row = blockIdx.x;  // (gidx, b, hq)
    const int hq = row % p.Hq;
    const int b = (row / p.Hq) % p.B;
    const int gidx = row / (p.Hq * p.B);
    const int layer = p.layer_of_global[gidx];
    const int e = threadIdx.x;
    const float* ml = p.ws_ml + static_cast<size_t>(row) * p.nsplit * 2;
    const float* os = p.ws_o + static_cast<size_t>(row) * p.nsplit * D;
    float mt = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) mt = fmaxf(mt, ml[2 * s]);
    float lt = 0.f, ot = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
        const float ms = ml[2 * s];
        if (ms == -INFINITY) continue;
        const float c = ex2_approx(ms - mt);
        lt += ml[2 * s + 1] * c;
        ot += os[static_cast<size_t>(s) * D + e] * c;
    }
    const size_t orow = (static_cast<size_t>(layer) * p.B + b) * p.Hq + hq;
    if (!idx_ok(p.ctl, static_cast<long long>(orow), static_cast<long long>(p.NL) * p.B * p.Hq, 76)) return;
    p.out[orow * D + e] = __float2bfloat16_rn(lt > 0.f ? ot / lt : 0.f);
}

template <int D, bool FP8, int NH>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
    using C = Dec<D, FP8>;
    auto kern = decode_attn_kernel<D, FP8, NH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.NG) * p.B * p.Hkv * p.nsplit +
                           static_cast<long long>(p.NS) * p.B * p.Hkv;
    if (ctas > 0) kern<<<static_cast<unsigned>(ctas), NTHR, C::SMEM, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.NG > 0) decode_combine_kernel<D><<<p.NG * p.B * p.Hq, D, 0, s>>>(p);
    return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_nh(const DecodeParams& p, cudaStream_t s) {
    return p.Hq / p.Hkv > 8 ? launch_t<D, FP8, 2>(p, s) : launch_t<D, FP8, 1>(p, s);
}

}  // namespace

size_t decode_workspace_bytes(int NG, int B, int Hq, int d, long long S) {
    const long long nsplit = (S + kDecodeSplitLen - 1) / kDecodeSplitLen;
    const size_t rows = static_cast<size_t>(NG) * B * Hq * nsplit;
    return rows * (static_cast<size_t>(d) + 2) * sizeof(float);
}

int decode_cache_box_rows(int d, bool fp8) { return static_cast<int>(STAGE_T) / (d * (fp8 ? 1 : 2)); }

bool decode_supports(int d, int G) { return (d == 64 || d == 128) && G >= 1 && G <= 16; }

cudaError_t launch_hybrid_decode(const DecodeParams& p, int d, cudaStream_t s) {
    if (p.Hkv <= 0 || p.Hq % p.Hkv || !decode_supports(d, p.Hq / p.Hkv)) return cudaErrorInvalidValue;
    if (d == 128) return p.fp8 ? launch_nh<128, true>(p, s) : launch_nh<128, false>(p, s);
    return p.fp8 ? launch_nh<64, true>(p, s) : launch_nh<64, false>(p, s);
}

}  // namespace zg
