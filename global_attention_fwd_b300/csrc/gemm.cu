// gemm.cu -- the projections of the gated sliding-window layer on the tensor cores, with the
// layer's element-wise work fused into the GEMM epilogue.
//
// "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ"; hyper.ai summary of
// arXiv 2609.13356, section "方法" (the GatedSWA equation):
//   q = h W_q, k = h W_k, v = h W_v, g = h W_g   (projections of the normalised hidden state)
//   a = A_SWA(q_hat, k_hat, v) * sigmoid(g),   y = a W_o
// with q_hat = RoPE(RMSNorm(q)), k_hat likewise (per head, QK norm + partial RoPE).
//
// One persistent kernel computes Y_i = X W_i for up to four weight matrices that share X (the
// four input projections in one launch, so h is read once), each with its own epilogue:
//   mode 0  Y = bf16(acc)                                     (v, and o_proj)
//   mode 1  Y = fp16(RoPE(RMSNorm(acc per head; w), pos))    (q_hat, k_hat: straight from the fp32
//           accumulator, so q and k are never rounded before the norm)
//   mode 2  Y = bf16(sigmoid(acc))                            (the gate, in fp32 without cancellation)
// X [M, K] and W_i [K, N_i] are bf16 row-major (y = x W); Y_i [M, N_i] row-major.
//
// Tiles of 128 rows x 256 columns, K in blocks of 64.  Warp roles (192 threads, one CTA per SM):
//   warp 0  TMA (one thread): X box {64 K, 128 rows} (K-major, 128-byte swizzle) and four W boxes
//           {64 N, 64 K} (MN-major) per stage into a 4-stage ring.
//   warp 1  MMA (one thread): tcgen05.mma kind::f16, M128 x N256 x K16, four per K block, into
//           one of two TMEM accumulators (256 columns each), so the epilogue of tile t overlaps
//           the products of tile t + 1.  Warp 1 owns TMEM (512 columns).
//   warps 2-5  epilogue: each reads its TMEM lane quarter (warp % 4), applies the mode, stores.
#include "zg_qk.cuh"

namespace zg {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;          // 16 KB
constexpr uint32_t kBBytes = kBK * kBN * 2;          // 32 KB: four 64-column boxes of 64 K rows
constexpr uint32_t kBChunk = kBK * 128;              // one 64-column box (64 rows x 128 B)
constexpr uint32_t kStageBytes = kABytes + kBBytes;  // 48 KB
constexpr int kRotStride = 65;                       // floats per row of the RoPE scratch (65: no bank conflicts)
constexpr uint32_t kOffRot = kStages * kStageBytes;  // [128 rows][65] fp32, one private row per epilogue thread
constexpr uint32_t kOffBar = kOffRot + 128 * kRotStride * 4;
constexpr uint32_t kSmem = kOffBar + 256;
static_assert(kSmem <= 232448, "shared memory budget");
constexpr int kThreads = 192;
constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, false, true);  // A K-major, B MN-major

struct TileCoord {
    int mi, ni, b;  // row tile, column tile within matrix b
};
constexpr int kGroupM = 16;  // row tiles per raster group
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, long long t) {
    // Column tiles of the matrices one after the other.  Tiles run in groups of kGroupM row tiles:
    // inside a group the row tile changes fastest, then the column tile, so the ~148 tiles in
    // flight at once cover about 16 row panels of X and 9 column panels of W, all resident in L2
    // (row tiles fastest over all rows would stream every row panel of X once per column panel).
    TileCoord c;
    const long long tn = p.tiles / p.tiles_m;  // column tiles over all matrices
    const long long per_group = static_cast<long long>(kGroupM) * tn;
    const int g = static_cast<int>(t / per_group);
    const int rows = min(kGroupM, p.tiles_m - g * kGroupM);
    const long long r = t - g * per_group;
    c.mi = g * kGroupM + static_cast<int>(r % rows);
    int n = static_cast<int>(r / rows);
    int b = 0;
    while (b + 1 < p.nb && n >= p.tiles_n[b]) n -= p.tiles_n[b++];
    c.ni = n;
    c.b = b;
    return c;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// eight 16-bit values (four packed words) to row-major global memory, 16-byte aligned
__device__ __forceinline__ void st8(void* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;  // [2] an accumulator holds a finished tile
    uint64_t* acc_empty = acc_full + 2;    // [2] the epilogue has read it (128 arrivals)
    uint64_t* drain = acc_empty + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (p.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 88, kErrAlign);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 128);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA (one thread)
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_a);
            for (int b = 0; b < p.nb; ++b) tma_prefetch_desc(&p.tm_b[b]);
            bool ok = true;
            int it = 0;  // K blocks issued so far (stage ring position)
            for (long long t = blockIdx.x; t < p.tiles && ok && !aborted(); t += gridDim.x) {
                const TileCoord c = tile_coord(p, t);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % kStages;
                    if (it >= kStages && !(ok = mbar_wait(&empty[s], ((it / kStages) - 1) & 1, p.ctl, 89))) break;
                    uint8_t* st = smem + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    tma_load_2d(st, &p.tm_a, &full[s], kb * kBK, c.mi * kBM);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch)
                        tma_load_2d(st + kABytes + ch * kBChunk, &p.tm_b[c.b], &full[s], c.ni * kBN + ch * 64, kb * kBK);
                }
            }
            if (!ok) fail();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA (one thread)
        if (lane == 0 && !aborted()) {
            bool ok = true;
            int it = 0, tl = 0;
            for (long long t = blockIdx.x; t < p.tiles && ok && !aborted(); t += gridDim.x, ++tl) {
                const int ab = tl & 1;
                if (tl >= 2 && !(ok = mbar_wait(&acc_empty[ab], ((tl >> 1) - 1) & 1, p.ctl, 90))) break;
                tc_fence_after();
                const uint32_t d = tbase + ab * kBN;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!(ok = mbar_wait(&full[s], (it / kStages) & 1, p.ctl, 91))) break;
                    tc_fence_after();
                    const uint64_t a0 = sdesc(sbase + s * kStageBytes, 16, 1024, kSw128);
                    const uint64_t b0 = sdesc(sbase + s * kStageBytes + kABytes, kBChunk, 1024, kSw128);
#pragma unroll
                    for (int ks = 0; ks < kBK / 16; ++ks)
                        umma_bf16(d, a0 + ((ks * 32) >> 4), b0 + ((ks * 16 * 128) >> 4), kIdesc, (kb | ks) != 0);
                    umma_commit(&empty[s]);  // the stage is free once these products have read it
                }
                umma_commit(&acc_full[ab]);
            }
            if (!ok) fail();
            umma_commit(drain);
            (void)mbar_wait(drain, 0, p.ctl, 92);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;
        const int rt = quarter * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
        const int half = p.rope.half;  // rotary pairs (j, j + half), half <= 32: inside the first 64 columns
        int tl = 0;
        for (long long t = blockIdx.x; t < p.tiles && !aborted(); t += gridDim.x, ++tl) {
            const TileCoord c = tile_coord(p, t);
            const int ab = tl & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (tl >> 1) & 1, p.ctl, 93))) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t acc = lane_addr + ab * kBN;
            const long long row = static_cast<long long>(c.mi) * kBM + rt;
            const bool row_ok = row < p.M;
            const int n = p.n[c.b], mode = p.mode[c.b];
            const int col0 = c.ni * kBN;
            uint16_t* yrow = static_cast<uint16_t*>(p.y[c.b]) + row * n;
            if (mode != 1) {
#pragma unroll 1
                for (int cb = 0; cb < kBN; cb += 32) {
                    uint32_t r[32];
                    tmem_ld32(acc + cb, r);
                    tmem_wait_ld();
                    if (!row_ok) continue;
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8) {
                        const int col = col0 + cb + 8 * g8;
                        if (col >= n) break;
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            float x0 = __uint_as_float(r[8 * g8 + 2 * k]), x1 = __uint_as_float(r[8 * g8 + 2 * k + 1]);
                            if (mode == 2) {
                                const float2 sg = sigmoid2_f32(make_float2(x0, x1));
                                x0 = sg.x;
                                x1 = sg.y;
                            }
                            w4[k] = pack_bf16x2(x0, x1);
                        }
                        st8(yrow + col, w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            } else {
                // per head of hd columns: RMSNorm over the head, weights, partial RoPE (rotate-half
                // pairs (j, j + half), j < half <= 32, all inside the head's first 64 columns), fp16
                const int hd = p.head_dim;
                const float* w = p.w[c.b];
                const int pos = row_ok ? __ldg(p.pos + row) : 0;
                float* xs = reinterpret_cast<float*>(smem + kOffRot) + rt * kRotStride;  // this row's scratch
#pragma unroll 1
                for (int hc = 0; hc < kBN; hc += hd) {
                    if (col0 + hc >= n) break;
                    float ss = 0.f;
#pragma unroll 1
                    for (int cb = 0; cb < hd; cb += 32) {
                        uint32_t r[32];
                        tmem_ld32(acc + hc + cb, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) ss = fmaf(__uint_as_float(r[k]), __uint_as_float(r[k]), ss);
                    }
                    const float inv = ss > 0.f || p.eps > 0.f ? rsqrtf(ss / hd + p.eps) : 0.f;
                    // the head's first 64 columns, normalised and weighted, through the row scratch
#pragma unroll 1
                    for (int cb = 0; cb < 64; cb += 32) {
                        uint32_t r[32];
                        tmem_ld32(acc + hc + cb, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) xs[cb + k] = __uint_as_float(r[k]) * inv * __ldg(w + cb + k);
                    }
#pragma unroll 1
                    for (int j = 0; j < half; ++j) {
                        float cj, sj;
                        rope_cos_sin(pos, p.rope.f_hi[j], p.rope.f_lo[j], cj, sj);
                        const float a2 = xs[j], b2 = xs[j + half];
                        xs[j] = a2 * cj - b2 * sj;
                        xs[j + half] = b2 * cj + a2 * sj;
                    }
                    if (row_ok) {
#pragma unroll
                        for (int g8 = 0; g8 < 8; ++g8)
                            st8(yrow + col0 + hc + 8 * g8, pack_half2(xs[8 * g8], xs[8 * g8 + 1]),
                                pack_half2(xs[8 * g8 + 2], xs[8 * g8 + 3]), pack_half2(xs[8 * g8 + 4], xs[8 * g8 + 5]),
                                pack_half2(xs[8 * g8 + 6], xs[8 * g8 + 7]));
                    }
                    if (hd > 64) {
#pragma unroll 1
                        for (int cb = 64; cb < hd; cb += 32) {
                            uint32_t r[32];
                            tmem_ld32(acc + hc + cb, r);
                            tmem_wait_ld();
                            if (!row_ok) continue;
#pragma unroll
                            for (int g8 = 0; g8 < 4; ++g8) {
                                uint32_t w4[4];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const int e = cb + 8 * g8 + 2 * k;
                                    w4[k] = pack_half2(__uint_as_float(r[8 * g8 + 2 * k]) * inv * __ldg(w + e),
                                                       __uint_as_float(r[8 * g8 + 2 * k + 1]) * inv * __ldg(w + e + 1));
                                }
                                st8(yrow + col0 + hc + cb + 8 * g8, w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[ab]);
        }
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        // abandoned run: give copies still in flight time to land before shared memory is released
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (p.tiles <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>(p.tiles < sms ? p.tiles : sms);
    gemm_kernel<<<grid, kThreads, kSmem, s>>>(p);
    return cudaGetLastError();
}

int gemm_tile_m() { return kBM; }
int gemm_tile_n() { return kBN; }

}  // namespace zg
