// hybrid_decode.cu -- one decode step through the hybrid 32-layer stack.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ": 27 local
// layers keep a KV cache of the last 128 tokens, the 5 global layers keep the
// whole sequence; decode is bound by memory bandwidth, so its cost is the cache
// it reads.  "ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for
// Math and Agentic Search" (jaehun.me review), section "KV 캐시가 6.4배 줄어드는
// 이유": 20 KiB of cache per token (5 global layers x 8 KV heads x 128 x K,V x
// bf16).
//
// Per layer l, sequence b, KV head g (4 query heads), new token at position p:
//   q_hat, k_hat = RoPE(RMSNorm(.)) at p; k_hat and v_new go to the cache
//   (global layer: slot p; local layer: ring slot p mod W); the 4 query heads
//   attend to positions 0..p (global) or max(0, p-W+1)..p (local, gated).
//
// Kernel 1 (attention, split-K).  One CTA per (global layer, b, g, split of
// 8192 keys) and per (local layer, b, g).  Warp 8 streams the cache slice into
// shared memory with 1-D bulk copies (cp.async.bulk, 32 keys = 16 KB of K and V
// per stage, six stages in flight); warps 0-7 consume it.  Half a warp handles one key:
// lane i holds 8 dims of q_hat for the 4 heads, reduces the 4 dot products with
// a 5-step recursive-halving shuffle, and keeps a per-head online softmax
// (max only raised when a score exceeds it by 8 in log2 units, so rescaling is
// rare) with packed fp32x2 FMAs.  Partials of the 16 key streams of the CTA are
// merged in shared memory; global splits write (m, l, o) to the workspace,
// local layers finish in place (1/l, sigmoid gate, bf16 store).  The CTA that
// owns position p also writes the new cache slot and adds the new key itself.
// Kernel 2 merges the splits of every global (layer, b, head) in a fixed order.
//
// FP8 caches use E4M3, the forward FP8 format of the training recipe in
// "ZGCM-1-7B 完全解説", section "学習の高速化 — FP8・Muon・TWEOが生む約4.2倍の効率".
// They hold e4m3(k_hat * k_scale) and e4m3(v * v_scale): the same stage bytes carry
// 64 keys instead of 32, lanes widen e4m3 pairs to fp16 pairs, 1 / k_scale is folded
// into q_hat and 1 / v_scale into the output.  RMSNorm bounds |k_hat| by sqrt(d) max|wk|,
// far inside the E4M3 range, so keys need no scale beyond that bound.
#include <cuda_fp8.h>

#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int D = 128;
constexpr int G = 4;               // query heads per KV head
constexpr int KPS = 32;            // keys per stage (bf16 caches; 64 for fp8 caches)
constexpr int NST = 6;             // stages (6 x 32 keys measured faster than 3 x 64 on B300)
constexpr int NCW = 8;             // compute warps
constexpr int NTHR = (NCW + 1) * 32;
constexpr uint32_t STAGE_K = KPS * D * 2;      // bytes of K per stage
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_V = NST * STAGE_K;
constexpr uint32_t OFF_QH = 2 * NST * STAGE_K;  // q_hat [4][128] f32
constexpr uint32_t OFF_KH = OFF_QH + G * D * 4;  // k_hat [128] f32
constexpr uint32_t OFF_VN = OFF_KH + D * 4;      // v_new [128] f32
constexpr uint32_t OFF_BAR = OFF_VN + D * 4;
constexpr uint32_t SMEM = OFF_BAR + 128;
static_assert(2 * NST * 8 + 4 <= 128, "barrier area");
constexpr float kLazy = 8.0f;  // raise the running max only past this margin (log2 units)

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
    unsigned long long r = *reinterpret_cast<unsigned long long*>(&acc);
    asm("fma.rn.f32x2 %0, %1, %2, %0;"
        : "+l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    acc = *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) { return make_float2(bf16lo(u), bf16hi(u)); }
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t u) {  // two E4M3 values, low byte first
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

template <bool FP8>
__global__ void __launch_bounds__(NTHR, 2) decode_attn_kernel(const __grid_constant__ DecodeParams p) {
    // 8 elements of a cache row (bf16: four words; E4M3: the first two words) -> 4 float pairs
    auto widen4 = [](const uint4& w, float2* f) {
        if (FP8) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                f[k] = e4m3x2_to_f2(static_cast<uint16_t>((k < 2 ? w.x : w.y) >> (16 * (k & 1))));
        } else {
            f[0] = bf2_to_f2(w.x);
            f[1] = bf2_to_f2(w.y);
            f[2] = bf2_to_f2(w.z);
            f[3] = bf2_to_f2(w.w);
        }
    };
    constexpr int EB = FP8 ? 1 : 2;        // bytes per cache element
    constexpr int KPT = FP8 ? 2 * KPS : KPS;  // keys per stage
    static_assert(KPT * D * EB == STAGE_K, "a stage holds the same bytes for either cache type");
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* empty = full + NST;
    int* sflag = reinterpret_cast<int*>(empty + NST);
    float* qh = reinterpret_cast<float*>(smem + OFF_QH);
    float* kh = reinterpret_cast<float*>(smem + OFF_KH);
    float* vn = reinterpret_cast<float*>(smem + OFF_VN);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- which work item
    const long long n_glob = static_cast<long long>(p.NG) * p.B * p.Hkv * p.nsplit;
    long long bid = blockIdx.x;
    bool is_glob = bid < n_glob;
    int layer, lidx, b, g, split = 0;
    if (is_glob) {
        split = static_cast<int>(bid % p.nsplit);
        long long r = bid / p.nsplit;
        g = static_cast<int>(r % p.Hkv);
        r /= p.Hkv;
        b = static_cast<int>(r % p.B);
        lidx = static_cast<int>(r / p.B);
        layer = p.layer_of_global[lidx];
    } else {
        long long r = bid - n_glob;
        g = static_cast<int>(r % p.Hkv);
        r /= p.Hkv;
        b = static_cast<int>(r % p.B);
        lidx = static_cast<int>(r / p.B);
        layer = p.layer_of_local[lidx];
    }
    const int pos = __ldg(p.pos + b);
    const bool pos_ok = pos >= 0 && static_cast<long long>(pos) < p.S;
    // keys streamed from the cache (positions before p) and whether this CTA owns p
    const uint8_t *kc, *vc;                       // cache rows of D elements, EB bytes each
    uint8_t *kslot = nullptr, *vslot = nullptr;
    int nk = 0;
    bool owner = false;
    if (is_glob) {
        const size_t base = ((static_cast<size_t>(lidx) * p.B + b) * p.Hkv + g) * static_cast<size_t>(p.S);
        const long long k0 = static_cast<long long>(split) * p.split_len;
        long long k1 = k0 + p.split_len;
        if (pos_ok && k1 > pos) k1 = pos;
        nk = pos_ok && k1 > k0 ? static_cast<int>(k1 - k0) : 0;
        kc = reinterpret_cast<const uint8_t*>(p.k_glob) + (base + k0) * D * EB;
        vc = reinterpret_cast<const uint8_t*>(p.v_glob) + (base + k0) * D * EB;
        owner = pos_ok && pos / p.split_len == split;
        kslot = reinterpret_cast<uint8_t*>(p.k_glob) + (base + pos) * D * EB;
        vslot = reinterpret_cast<uint8_t*>(p.v_glob) + (base + pos) * D * EB;
    } else {
        const size_t base = ((static_cast<size_t>(lidx) * p.B + b) * p.Hkv + g) * static_cast<size_t>(p.W);
        nk = pos_ok ? p.W : 0;  // every slot is streamed; invalid ones are masked below
        kc = reinterpret_cast<const uint8_t*>(p.k_ring) + base * D * EB;
        vc = reinterpret_cast<const uint8_t*>(p.v_ring) + base * D * EB;
        owner = pos_ok;
        kslot = reinterpret_cast<uint8_t*>(p.k_ring) + (base + (pos_ok ? pos % p.W : 0)) * D * EB;
        vslot = reinterpret_cast<uint8_t*>(p.v_ring) + (base + (pos_ok ? pos % p.W : 0)) * D * EB;
    }
    const int nstage = (nk + KPT - 1) / KPT;

    if (threadIdx.x == 0) {
        *sflag = 1;
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ---------------- producer: stream the cache slice
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int st = 0; st < nstage && ok; ++st) {
                const int buf = st % NST;
                ok = mbar_wait(&empty[buf], ((st / NST) & 1) ^ 1, p.ctl, 40);
                if (!ok) break;
                const int rows = min(KPT, nk - st * KPT);
                mbar_arrive_expect_tx(&full[buf], 2u * rows * D * EB);
                bulk_load(smem + OFF_K + buf * STAGE_K, kc + static_cast<size_t>(st) * KPT * D * EB, rows * D * EB,
                          &full[buf]);
                bulk_load(smem + OFF_V + buf * STAGE_K, vc + static_cast<size_t>(st) * KPT * D * EB, rows * D * EB,
                          &full[buf]);
                ++issued;
            }
            if (!ok) {
                *sflag = 0;
                // drain: every issued copy must land before the CTA may exit
                for (int st = max(0, issued - NST); st < issued; ++st)
                    (void)mbar_wait(&full[st % NST], (st / NST) & 1, p.ctl, 41);
            }
        }
    } else if (warp < G + 1) {
        // ---------------- q_hat for the 4 heads (warps 0-3), k_hat / v_new (warp 4)
        if (pos_ok) {
            const size_t tok = static_cast<size_t>(layer) * p.B + b;
            if (warp < G) {
                norm_rope_warp(p.q + (tok * p.Hq + g * G + warp) * D, p.wq + static_cast<size_t>(layer) * D, p.eps,
                               pos, p.rope, p.scale_log2, qh + warp * D);
            } else if (owner) {
                const __nv_bfloat16* kn = p.k_new + (tok * p.Hkv + g) * D;
                norm_rope_warp(kn, p.wk + static_cast<size_t>(layer) * D, p.eps, pos, p.rope, 1.0f, kh);
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
        }
    }
    // compute warps wait for q_hat (named barrier over the 8 compute warps)
    if (warp < NCW) asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");

    // per-lane state: 8 dims (dslice) of every head; half-warp hw handles every other key
    const int hw = lane >> 4;
    const int dl = (lane & 15) * 8;
    float2 qv[G][4];
    float m[G], l[G];
    float2 o[G][4];
    const float qs = FP8 ? 1.0f / p.k_scale : 1.0f;  // scores of stored keys come out unscaled
    const float vs = FP8 ? p.v_scale : 1.0f;         // stored values are v * vs
    if (warp < NCW) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qv[h][k] = make_float2(qh[h * D + dl + 2 * k] * qs, qh[h * D + dl + 2 * k + 1] * qs);
                o[h][k] = make_float2(0.f, 0.f);
            }
            m[h] = -INFINITY;
            l[h] = 0.f;
        }
        const bool ring = !is_glob;
        const int wslot = pos_ok ? pos % p.W : -1;
        bool ok = true;
        for (int st = 0; st < nstage; ++st) {
            const int buf = st % NST;
            ok = ok && *sflag && mbar_wait(&full[buf], (st / NST) & 1, p.ctl, 42);
            if (!ok) break;
            const uint8_t* sk = smem + OFF_K + buf * STAGE_K;
            const uint8_t* sv = smem + OFF_V + buf * STAGE_K;
#pragma unroll 2
            for (int it = 0; it < KPT / (NCW * 2); ++it) {
                const int kr = warp * (KPT / NCW) + it * 2 + hw;  // key row within the stage
                const int key = st * KPT + kr;
                bool valid = key < nk;
                if (ring) valid = valid && key != wslot && (pos >= p.W - 1 || key < pos);
                // raw words now, widened where they are used (keeps the live registers down)
                uint4 kraw, vraw;
                if (FP8) {
                    const uint2 kq = *reinterpret_cast<const uint2*>(sk + kr * D + dl);
                    const uint2 vq = *reinterpret_cast<const uint2*>(sv + kr * D + dl);
                    kraw = make_uint4(kq.x, kq.y, 0u, 0u);
                    vraw = make_uint4(vq.x, vq.y, 0u, 0u);
                } else {
                    kraw = *reinterpret_cast<const uint4*>(sk + kr * (D * 2) + dl * 2);
                    vraw = *reinterpret_cast<const uint4*>(sv + kr * (D * 2) + dl * 2);
                }
                float2 k2[4];
                widen4(kraw, k2);
                float part[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k = 0; k < 4; ++k) ffma2(acc, qv[h][k], k2[k]);
                    part[h] = acc.x + acc.y;
                }
                // recursive halving over the 16 lanes of the key: lane keeps head (lane>>2)&3
                {
                    const bool up8 = lane & 8;
                    float a0 = up8 ? part[0] : part[2], a1 = up8 ? part[1] : part[3];
                    float k0v = up8 ? part[2] : part[0], k1v = up8 ? part[3] : part[1];
                    k0v += __shfl_xor_sync(0xffffffffu, a0, 8);
                    k1v += __shfl_xor_sync(0xffffffffu, a1, 8);
                    const bool up4 = lane & 4;
                    float keep = up4 ? k1v : k0v;
                    keep += __shfl_xor_sync(0xffffffffu, up4 ? k0v : k1v, 4);
                    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
                    keep += __shfl_xor_sync(0xffffffffu, keep, 1);
                    // lane holds the score of head ((lane>>3)&1)*2 + ((lane>>2)&1); gather all four
                    const int src = lane & 16;
                    part[0] = __shfl_sync(0xffffffffu, keep, src + 0);
                    part[1] = __shfl_sync(0xffffffffu, keep, src + 4);
                    part[2] = __shfl_sync(0xffffffffu, keep, src + 8);
                    part[3] = __shfl_sync(0xffffffffu, keep, src + 12);
                }
                float2 v2[4];
                widen4(vraw, v2);
                if (valid) {
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float s = part[h];
                        if (s > m[h] + kLazy || m[h] == -INFINITY) {
                            const float corr = m[h] == -INFINITY ? 0.f : ex2_approx(m[h] - s);
                            m[h] = s;
                            l[h] *= corr;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                o[h][k].x *= corr;
                                o[h][k].y *= corr;
                            }
                        }
                        const float pr = ex2_approx(s - m[h]);
                        l[h] += pr;
                        const float2 p2 = make_float2(pr, pr);
#pragma unroll
                        for (int k = 0; k < 4; ++k) ffma2(o[h][k], p2, v2[k]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[buf]);
        }
        if (!ok) *sflag = 0;
        // the new key (owner only), handled by half-warp 0 of warp 0
        if (owner && warp == 0 && hw == 0 && ok) {
            float part[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = fmaf(qh[h * D + dl + k], kh[dl + k], acc);
#pragma unroll
                for (int off = 8; off; off >>= 1) acc += __shfl_xor_sync(0x0000ffffu, acc, off);
                part[h] = acc;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float s = part[h];
                if (s > m[h]) {
                    const float corr = m[h] == -INFINITY ? 0.f : ex2_approx(m[h] - s);
                    m[h] = s;
                    l[h] *= corr;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        o[h][k].x *= corr;
                        o[h][k].y *= corr;
                    }
                }
                const float pr = ex2_approx(s - m[h]);
                l[h] += pr;
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // in the units of the stored values
                    o[h][k].x = fmaf(pr, vn[dl + 2 * k] * vs, o[h][k].x);
                    o[h][k].y = fmaf(pr, vn[dl + 2 * k + 1] * vs, o[h][k].y);
                }
            }
        }
        // merge the two half-warps (same dims, different keys)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[h], 16);
            const float lo = __shfl_xor_sync(0xffffffffu, l[h], 16);
            const float mt = fmaxf(m[h], mo);
            const float c0 = m[h] == -INFINITY ? 0.f : ex2_approx(m[h] - mt);
            const float c1 = mo == -INFINITY ? 0.f : ex2_approx(mo - mt);
            l[h] = l[h] * c0 + lo * c1;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float ox = __shfl_xor_sync(0xffffffffu, o[h][k].x, 16);
                const float oy = __shfl_xor_sync(0xffffffffu, o[h][k].y, 16);
                o[h][k].x = o[h][k].x * c0 + ox * c1;
                o[h][k].y = o[h][k].y * c0 + oy * c1;
            }
            m[h] = mt;
        }
    }
    __syncthreads();  // every stage consumed, every copy landed: stage buffers are free

    // ---- merge the 8 warps in shared memory (reuses the K stage area)
    float* red_o = reinterpret_cast<float*>(smem + OFF_K);          // [NCW][G][D]
    float* red_ml = reinterpret_cast<float*>(smem + OFF_V);         // [NCW][G][2]
    if (warp < NCW && hw == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                red_o[(warp * G + h) * D + dl + 2 * k] = o[h][k].x;
                red_o[(warp * G + h) * D + dl + 2 * k + 1] = o[h][k].y;
            }
            if (lane == 0) {
                red_ml[(warp * G + h) * 2 + 0] = m[h];
                red_ml[(warp * G + h) * 2 + 1] = l[h];
            }
        }
    }
    __syncthreads();
    const bool all_ok = *sflag != 0;
    for (int idx = threadIdx.x; idx < G * D; idx += NTHR) {
        const int h = idx / D, e = idx % D;
        float mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) mt = fmaxf(mt, red_ml[(w * G + h) * 2]);
        float lt = 0.f, ot = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = red_ml[(w * G + h) * 2];
            const float c = mw == -INFINITY ? 0.f : ex2_approx(mw - mt);
            lt += red_ml[(w * G + h) * 2 + 1] * c;
            ot += red_o[(w * G + h) * D + e] * c;
        }
        ot *= 1.0f / vs;
        const int hq = g * G + h;
        if (is_glob) {
            const size_t row = ((static_cast<size_t>(lidx) * p.B + b) * p.Hq + hq) * p.nsplit + split;
            p.ws_o[row * D + e] = (all_ok ? ot : 0.f);
            if (e == 0) {
                p.ws_ml[row * 2 + 0] = all_ok ? mt : -INFINITY;
                p.ws_ml[row * 2 + 1] = all_ok ? lt : 0.f;
            }
        } else {
            const size_t orow = (static_cast<size_t>(layer) * p.B + b) * p.Hq + hq;
            float r = 0.f;
            if (all_ok && lt > 0.f) {
                const float gt = __bfloat162float(p.gate[orow * D + e]);
                r = ot / lt * sigmoid_f32(gt);
            }
            p.out[orow * D + e] = __float2bfloat16_rn(r);
        }
    }
}

// merge the splits of one (global layer, b, query head): 128 threads, one per dim
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
    p.out[orow * D + e] = __float2bfloat16_rn(lt > 0.f ? ot / lt : 0.f);
}

}  // namespace

size_t decode_workspace_bytes(int NG, int B, int Hq, long long S) {
    const long long nsplit = (S + kDecodeSplitLen - 1) / kDecodeSplitLen;
    const size_t rows = static_cast<size_t>(NG) * B * Hq * nsplit;
    return rows * (D + 2) * sizeof(float);
}

cudaError_t launch_hybrid_decode(const DecodeParams& p, int d, cudaStream_t s) {
    if (d != D || p.Hq != p.Hkv * G) return cudaErrorInvalidValue;
    auto kern = p.fp8 ? decode_attn_kernel<true> : decode_attn_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.NG) * p.B * p.Hkv * p.nsplit +
                           static_cast<long long>(p.NS) * p.B * p.Hkv;
    if (ctas > 0) kern<<<static_cast<unsigned>(ctas), NTHR, SMEM, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.NG > 0) decode_combine_kernel<<<p.NG * p.B * p.Hq, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
