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
// Kernel 1 (prep, four rows per warp): q_hat, k_hat and dA = dout * sigmoid(gate) in bf16.
//
// Kernel 2 (query pass): one CTA per tile of 32 tokens x the 4 query heads of one KV
// head (128 rows); the tile sees the 160 keys [t0 - 128, t0 + 32).
//   warp 8 (one thread): TMA of Q_hat, dA, K_hat, V; the MMAs
//     S = Q_hat K_hat^T  (N = 160)  -> TMEM [0, 160)
//     dP = dA V^T        (N = 160)  -> TMEM [160, 320)
//     O = P V   (P from TMEM, packed over S)          -> TMEM [320, 448)
//     dQ_hat = dS K_hat  (dS from TMEM, packed over dP) -> TMEM [320, 448) (after O is read)
//   warps 0-7 (thread = row = TMEM lane, two warps per row, one per column half): exact
//   row max and sum over the window, P
//   (unnormalised, bf16) over S; A = O / l, D, dgate = dA * A * (1 - sigmoid(gate)) and
//   the row statistics (max, 1 / l, D) for kernel 3; dS over dP; finally dQ_hat back
//   through RoPE and RMSNorm into dq (fp32).  Gate and dout tiles are staged by TMA into
//   Q_hat / dA once the first two products are done; dgate and dq leave through swizzled
//   fp32 staging tiles and bulk tensor stores.
//
// Kernel 3 (key pass): one CTA per 128 keys of one KV head; the queries that see them
// are the tokens [j0, j0 + 128 + W - 1), visited as query tiles of 32 tokens x 4 heads
// whose Q_hat / dA arrive on a two-stage TMA ring.
//   warp 4: S^T = K_hat Q_hat^T -> [0, 128), dP^T = V dA^T -> [128, 256), then
//     dV += P^T dA -> [256, 384), dK_hat += dS^T Q_hat -> [384, 512)
//     (P^T, dS^T from TMEM, packed over S^T and dP^T; one thread's MMAs run in issue
//     order, so the next tile's S^T overwrites P^T only after dV has read it).
//   warps 0-3 (thread = key row, query columns 0-63) and warps 4-7 (columns 64-127): P^T
//   and dS^T from the row statistics of kernel 2; the products of each column half are
//   issued separately, so one half's accumulation runs while the other half's rows are
//   computed.  At the end dV (fp32) and dK_hat back through RoPE and RMSNorm into dk, both
//   through swizzled fp32 staging tiles and bulk tensor stores.
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

// query pass shared memory: Q_hat, dA (later the gate and dout tiles), V, K_hat, raw q,
// the second half's dgate staging, the pair-exchange slots, wq
constexpr uint32_t QP_Q = 0;
constexpr uint32_t QP_DA = QP_Q + TILE128;
constexpr uint32_t QP_V = QP_DA + TILE128;
constexpr uint32_t QP_K = QP_V + TILE160;
constexpr uint32_t QP_X = QP_K + TILE160;
constexpr uint32_t QP_DG1 = QP_X + TILE128;          // dgate staging of column half 1 (two boxes)
constexpr uint32_t QP_XCH = QP_DG1 + 2 * 128 * 128;  // [2 parities][2 halves][128 rows] float2
constexpr uint32_t QP_W = QP_XCH + 2 * 2 * 128 * 8;
constexpr uint32_t QP_BAR = QP_W + D * 4;
constexpr int QP_NBAR = 64;
constexpr uint32_t QP_MISC = QP_BAR + QP_NBAR * 8;
constexpr uint32_t QP_SMEM = QP_MISC + 32;
constexpr uint32_t QP_DG0 = QP_V;   // dgate staging of column half 0 (two boxes) in the free V tile
constexpr uint32_t QP_DQ = QP_Q;    // dq staging (four boxes) over the free Q_hat and dA tiles
constexpr uint32_t QP_ROPE = QP_K;  // [T tokens][kMaxRotHalf] float2 in the free K_hat tile, at the end
static_assert(QP_DG0 + 2 * 128 * 128 <= QP_K && QP_DQ + 4 * 128 * 128 <= QP_DG0, "staging tiles");
static_assert(QP_ROPE + T * kMaxRotHalf * 8 <= QP_X, "RoPE table inside the K_hat tile");
static_assert(QP_K % 1024 == 0 && QP_V % 1024 == 0 && QP_X % 1024 == 0 && QP_DG1 % 1024 == 0, "swizzle atoms");
static_assert(QP_SMEM <= 227 * 1024, "shared memory");

// key pass shared memory
constexpr uint32_t KP_K = 0;
constexpr uint32_t KP_V = KP_K + TILE128;
constexpr uint32_t KP_QD = KP_V + TILE128;      // 2 stages x (Q_hat, dA)
constexpr uint32_t KP_STAT = KP_QD + 4 * TILE128;  // 8 warps x 64 float4
constexpr uint32_t KP_W = KP_STAT + 8 * 64 * 16;
constexpr uint32_t KP_BAR = KP_W + D * 4;
constexpr uint32_t KP_MISC = KP_BAR + 16 * 8;
constexpr uint32_t KP_SMEM = KP_MISC + 32;
constexpr uint32_t KP_X = KP_QD + 3 * TILE128;  // raw k tile, loaded into the free ring at the end
constexpr uint32_t KP_DV = KP_K;    // dv staging (four 32-column fp32 boxes) over K_hat and V
constexpr uint32_t KP_DK = KP_QD;   // dk staging over the first half of the query ring
static_assert(KP_DV + 4 * 128 * 128 <= KP_QD && KP_DK + 4 * 128 * 128 <= KP_X, "staging tiles");
static_assert(KP_SMEM <= 227 * 1024, "shared memory");

// 16-byte group c8 (elements 8 c8 .. 8 c8 + 7) of row r of a 128-row tile of two 64-column
// chunks with the 128-byte swizzle (the layout the TMA boxes land in)
__device__ __forceinline__ uint4 ld_row8(const uint8_t* tile, int r, int c8) {
    return *reinterpret_cast<const uint4*>(tile + (c8 >> 3) * CH128 + sw128_off(r, c8 & 7));
}

// A 128-row fp32 staging tile laid out as four boxes of 32 columns (128 rows x 128 bytes each)
// with the 128-byte swizzle: the layout a bulk tensor store of box {32, ...} reads.
constexpr uint32_t F32BOX = 128 * 128;
constexpr uint32_t F32TILE = 4 * F32BOX;
__device__ __forceinline__ float* f32_elem(uint8_t* t, int r, int e) {
    return reinterpret_cast<float*>(t + (e >> 5) * F32BOX + r * 128 + ((((e & 31) >> 2) ^ (r & 7)) << 4) + (e & 3) * 4);
}
__device__ __forceinline__ float4* f32_chunk(uint8_t* t, int r, int c4) {  // floats 4 c4 .. 4 c4 + 3 of row r
    return reinterpret_cast<float4*>(t + (c4 >> 3) * F32BOX + r * 128 + (((c4 & 7) ^ (r & 7)) << 4));
}

// One row, held by one thread in a staging tile: dy (the gradient of x_hat) in, the gradient of
// the raw row x out, in place.  RoPE rotated (a, b) by +angle, so its transpose rotates by
// -angle; RMSNorm x_hat = x * inv * w with inv = (mean x^2 + eps)^-1/2 gives
// dx = inv * w * dy - inv^3 / d * x * sum(x * w * dy).
// x: row r of a bf16 swizzled tile in shared memory; cos_sin(j) gives (cos, sin) of pair j.
template <class CosSin>
__device__ __forceinline__ void row_norm_rope_bwd(uint8_t* t, int r, const uint8_t* xtile, const float* w_s, float eps,
                                                  int half, CosSin cos_sin) {
    for (int j = 0; j < half; ++j) {
        const float2 c = cos_sin(j);
        float* pa = f32_elem(t, r, j);
        float* pb = f32_elem(t, r, j + half);
        const float a = *pa, bb = *pb;
        *pa = a * c.x + bb * c.y;
        *pb = bb * c.x - a * c.y;
    }
    float ss = 0.f, tw = 0.f;
#pragma unroll 4
    for (int c8 = 0; c8 < D / 8; ++c8) {
        const uint4 u = ld_row8(xtile, r, c8);
        const float4 y0 = *f32_chunk(t, r, 2 * c8), y1 = *f32_chunk(t, r, 2 * c8 + 1);
        const float x[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                            bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
        const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ss = fmaf(x[e], x[e], ss);
            tw = fmaf(x[e] * w_s[8 * c8 + e], y[e], tw);
        }
    }
    const float inv = ss > 0.f || eps > 0.f ? rsqrtf(ss * (1.0f / D) + eps) : 0.f;
    const float coef = inv * inv * inv * tw * (1.0f / D);
#pragma unroll 4
    for (int c8 = 0; c8 < D / 8; ++c8) {
        const uint4 u = ld_row8(xtile, r, c8);
        float4* p0 = f32_chunk(t, r, 2 * c8);
        float4* p1 = f32_chunk(t, r, 2 * c8 + 1);
        const float4 y0 = *p0, y1 = *p1;
        const float* w = w_s + 8 * c8;
        *p0 = make_float4(inv * w[0] * y0.x - coef * bf16lo(u.x), inv * w[1] * y0.y - coef * bf16hi(u.x),
                          inv * w[2] * y0.z - coef * bf16lo(u.y), inv * w[3] * y0.w - coef * bf16hi(u.y));
        *p1 = make_float4(inv * w[4] * y1.x - coef * bf16lo(u.z), inv * w[5] * y1.y - coef * bf16hi(u.z),
                          inv * w[6] * y1.z - coef * bf16lo(u.w), inv * w[7] * y1.w - coef * bf16hi(u.w));
    }
}

// TMEM columns [col, col + 128) of this thread's lane, times `scale`, into row r of a staging tile
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, uint8_t* t, int r, float scale) {
#pragma unroll 1
    for (int k = 0; k < D / 32; ++k) {
        uint32_t v[32];
        tmem_ld32(taddr + 32 * k, v);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *f32_chunk(t, r, 8 * k + c) =
                make_float4(__uint_as_float(v[4 * c]) * scale, __uint_as_float(v[4 * c + 1]) * scale,
                            __uint_as_float(v[4 * c + 2]) * scale, __uint_as_float(v[4 * c + 3]) * scale);
    }
}

// ---------------------------------------------------------------- kernel 1
// Four rows per warp (the q rows first, then the k rows), every global load issued before
// any arithmetic so that a warp keeps several rows in flight.
constexpr int kPrepRows = 4;

__global__ void __launch_bounds__(256) bwd_tc_prep_kernel(const __grid_constant__ BackwardTcParams p) {
    __shared__ float buf[8][kPrepRows][D];
    __shared__ float rope_f[2][kMaxRotHalf];  // read by lane-dependent index: staged out of the parameters
    stage_rope(p.rope, rope_f[0], rope_f[1]);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // row indices in 32-bit arithmetic: the host takes this path only for B * L * (Hq + Hkv) < 2^31
    const unsigned nq = static_cast<unsigned>(p.B * p.L) * p.Hq, nk = static_cast<unsigned>(p.B * p.L) * p.Hkv;
    const unsigned row0 = static_cast<unsigned>(p.prep_first) + (blockIdx.x * 8u + warp) * kPrepRows;
    const bool gated = p.gate != nullptr;
    uint2 xr[kPrepRows], gr[kPrepRows], dr[kPrepRows];
    int pos[kPrepRows];
#pragma unroll
    for (int i = 0; i < kPrepRows; ++i) {
        const unsigned row = row0 + i;
        const bool is_q = row < nq;
        const unsigned r = is_q ? row : row - nq;
        const bool valid = row < nq + nk;
        xr[i] = valid ? *reinterpret_cast<const uint2*>((is_q ? p.q : p.k) + static_cast<size_t>(r) * D + lane * 4)
                      : make_uint2(0u, 0u);
        const unsigned tok = r / static_cast<unsigned>(is_q ? p.Hq : p.Hkv);
        pos[i] = valid && idx_ok(p.ctl, tok, static_cast<long long>(p.B) * p.L, 150) ? __ldg(p.pos + tok) : 0;
        if (valid && is_q && gated) {
            gr[i] = *reinterpret_cast<const uint2*>(p.gate + static_cast<size_t>(r) * D + lane * 4);
            dr[i] = *reinterpret_cast<const uint2*>(p.dout + static_cast<size_t>(r) * D + lane * 4);
        }
    }
#pragma unroll
    for (int i = 0; i < kPrepRows; ++i) {
        const unsigned row = row0 + i;
        const bool is_q = row < nq;
        const float4 w = __ldg(reinterpret_cast<const float4*>((is_q ? p.wq : p.wk) + lane * 4));
        const float v0 = bf16lo(xr[i].x), v1 = bf16hi(xr[i].x), v2 = bf16lo(xr[i].y), v3 = bf16hi(xr[i].y);
        float ss = v0 * v0 + v1 * v1 + v2 * v2 + v3 * v3;
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = ss > 0.f || p.eps > 0.f ? rsqrtf(ss * (1.0f / D) + p.eps) : 0.f;
        *reinterpret_cast<float4*>(&buf[warp][i][lane * 4]) =
            make_float4(v0 * inv * w.x, v1 * inv * w.y, v2 * inv * w.z, v3 * inv * w.w);
    }
    __syncwarp();
    // rotate the pairs (j, j + half) of every row
    for (int j = lane; j < p.rope.half; j += 32) {
#pragma unroll
        for (int i = 0; i < kPrepRows; ++i) {
            float cs, sn;
            rope_cos_sin(pos[i], rope_f[0][j], rope_f[1][j], cs, sn);
            const float a = buf[warp][i][j], bb = buf[warp][i][j + p.rope.half];
            buf[warp][i][j] = a * cs - bb * sn;
            buf[warp][i][j + p.rope.half] = bb * cs + a * sn;
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kPrepRows; ++i) {
        const unsigned row = row0 + i;
        if (row >= nq + nk) break;
        const bool is_q = row < nq;
        const size_t r = is_q ? row : row - nq;
        const float4 v = *reinterpret_cast<const float4*>(&buf[warp][i][lane * 4]);
        *reinterpret_cast<uint2*>((is_q ? p.qh : p.kh) + r * D + lane * 4) =
            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        if (is_q && gated) {
            // the same sigmoid as the query pass, which rebuilds these bf16 values for D
            const uint2 go = gr[i], dd = dr[i];
            *reinterpret_cast<uint2*>(p.da + r * D + lane * 4) = make_uint2(
                pack_bf16x2(bf16lo(dd.x) * sigmoid_f32(bf16lo(go.x)), bf16hi(dd.x) * sigmoid_f32(bf16hi(go.x))),
                pack_bf16x2(bf16lo(dd.y) * sigmoid_f32(bf16lo(go.y)), bf16hi(dd.y) * sigmoid_f32(bf16hi(go.y))));
        }
    }
}

// ---------------------------------------------------------------- kernel 2: query pass
// Warps 0-7 own the rows two warps per TMEM lane quarter: warp w has the rows of quarter
// w & 3 and the column half w >> 2 (keys [80 h, 80 h + 80) of the score tiles, columns
// [64 h, 64 h + 64) of O and dQ_hat).  The two warps of a quarter exchange row partials
// (max, sum, D, RMSNorm sums) through shared memory and a 64-arrival barrier per exchange.
// Warp 8: TMA and MMA.
constexpr int kQThreads = 288;
constexpr int kNX = 8;  // pair exchange slots per tile (0-5, and 7 for the RMSNorm sums of the q_hat fold)

__global__ void __launch_bounds__(kQThreads, 1) bwd_qpass_kernel(const __grid_constant__ BackwardTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + QP_BAR);
    uint64_t* ld_full = bar + 0;
    uint64_t* s_full = bar + 1;
    uint64_t* p_ready = bar + 2;
    uint64_t* o_full = bar + 3;
    uint64_t* ds_ready = bar + 4;
    uint64_t* dq_full = bar + 5;
    uint64_t* gd_full = bar + 6;   // gate and dout tiles (gated layers)
    uint64_t* stg_full = bar + 7;  // [2] dgate staging of a column half written (128 arrivals)
    uint64_t* dq_stg = bar + 9;    // dq staging written (256 arrivals)
    uint64_t* qd_ready = bar + 10; // fold: q_hat and dA are in shared memory (256 arrivals)
    uint64_t* xbar = bar + 16;     // [kNX][4 quarters] pair exchanges (64 arrivals)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + QP_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + QP_MISC + 4);
    float* w_s = reinterpret_cast<float*>(smem + QP_W);
    float2* xch = reinterpret_cast<float2*>(smem + QP_XCH);
    constexpr uint32_t C_S = 0, C_DP = NKQ, C_O = 2 * NKQ;
    static_assert(16 + kNX * 4 <= QP_NBAR, "barrier slots");

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
        mbar_init(p_ready, 256);
        mbar_init(o_full, 1);
        mbar_init(ds_ready, 256);
        mbar_init(dq_full, 1);
        mbar_init(gd_full, 1);
        mbar_init(&stg_full[0], 128);
        mbar_init(&stg_full[1], 128);
        mbar_init(dq_stg, 256);
        mbar_init(qd_ready, 256);
        for (int i = 0; i < kNX * 4; ++i) mbar_init(&xbar[i], 64);
        fence_barrier_init();
    }
    if (threadIdx.x < 32)
        *reinterpret_cast<float4*>(w_s + lane * 4) = __ldg(reinterpret_cast<const float4*>(p.wq + lane * 4));
    const bool gated = p.gate != nullptr;
    if (warp == 8) {
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
    // TMEM column of the packed 16-bit operand for keys [16 ks, 16 ks + 16): each column half
    // packs its 80 keys into the first 40 columns of its own 80-column region
    auto packed_col = [](uint32_t base, int ks) { return base + 80 * (ks / 5) + 8 * (ks % 5); };

    if (warp == 8) {
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_qh);
            tma_prefetch_desc(&p.tm_da);
            tma_prefetch_desc(&p.tm_kq);
            tma_prefetch_desc(&p.tm_vq);
            tma_prefetch_desc(&p.tm_q);
            // fold: the gate (gated layers) and dout tiles instead of q_hat and dA, which the rows form
            const bool q_tile = !p.fold || gated;
            mbar_arrive_expect_tx(ld_full, (q_tile ? 3 : 2) * TILE128 + 2 * TILE160);
            for (int ch = 0; ch < 2; ++ch) {
                if (q_tile)
                    tma_load_4d(smem + QP_Q + ch * CH128, p.fold ? &p.tm_gate : &p.tm_qh, ld_full, ch * 64, g * G, t0, b);
                tma_load_4d(smem + QP_DA + ch * CH128, p.fold && gated ? &p.tm_dout : &p.tm_da, ld_full, ch * 64, g * G,
                            t0, b);
                tma_load_4d(smem + QP_K + ch * CH160, &p.tm_kq, ld_full, ch * 64, g, t0 - 128, b);
                tma_load_4d(smem + QP_V + ch * CH160, &p.tm_vq, ld_full, ch * 64, g, t0 - 128, b);
                tma_load_4d(smem + QP_X + ch * CH128, &p.tm_q, ld_full, ch * 64, g * G, t0, b);
            }
            constexpr uint32_t id_s = idesc_bf16_f32(128, NKQ, false, false);
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, false, true);
            bool ok = mbar_wait(ld_full, 0, p.ctl, 101);
            if (ok && p.fold) {
                // the rows' q_hat (and dA) go to the workspace for the key pass, read from shared memory
                // beside the first products; dout is the caller's tensor and is never written
                ok = mbar_wait(qd_ready, 0, p.ctl, 109);
                if (ok) {
                    for (int ch = 0; ch < 2; ++ch) {
                        tma_store_4d(&p.tm_qh, smem + QP_Q + ch * CH128, ch * 64, g * G, t0, b);
                        if (gated) tma_store_4d(&p.tm_da, smem + QP_DA + ch * CH128, ch * 64, g * G, t0, b);
                    }
                    bulk_commit();
                }
            }
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
                if (gated) {  // Q_hat and dA are read once the two products are done: reuse them
                    ok = mbar_wait(s_full, 0, p.ctl, 107);
                    if (ok && p.fold) bulk_wait_all();  // and once their stores have read them
                    if (ok) {
                        mbar_arrive_expect_tx(gd_full, 2 * TILE128);
                        for (int ch = 0; ch < 2; ++ch) {
                            tma_load_4d(smem + QP_Q + ch * CH128, &p.tm_gate, gd_full, ch * 64, g * G, t0, b);
                            tma_load_4d(smem + QP_DA + ch * CH128, &p.tm_dout, gd_full, ch * 64, g * G, t0, b);
                        }
                    }
                }
                if (ok) ok = mbar_wait(p_ready, 0, p.ctl, 102);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < NKQ / 16; ++ks)
                    umma_tmem_a(tbase + C_O, packed_col(tbase + C_S, ks),
                                sdesc(sbase + QP_V + ks * 16 * 128, CH160, 1024, kSw128), id_o, ks > 0);
                umma_commit(o_full);
                ok = mbar_wait(ds_ready, 0, p.ctl, 103);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < NKQ / 16; ++ks)
                    umma_tmem_a(tbase + C_O, packed_col(tbase + C_DP, ks),
                                sdesc(sbase + QP_K + ks * 16 * 128, CH160, 1024, kSw128), id_o, ks > 0);
                umma_commit(dq_full);
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ rows (thread = row = TMEM lane)
        const int q4 = warp & 3, hf = warp >> 2;
        const int row = q4 * 32 + lane;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q4 * 32) << 16);
        const int tt = row / G;
        const int t = t0 + tt;
        const bool valid_row = t < p.L;
        const long long qrow = (static_cast<long long>(b) * p.L + t) * p.Hq + g * G + row % G;
        const int lo = max(128 - t0, tt + 128 - p.window + 1);  // key columns [lo, hi] are in the window
        const int hi = tt + 128;
        const float sl = p.scale_log2;
        const int c0 = 80 * hf;  // this warp's key columns [c0, c0 + 80)
        // pair exchange k: publish a float pair, wait for the partner, return its pair.  Every
        // thread arrives at every exchange, so a partner that gave up never leaves this one
        // blocked longer than the bounded wait.
        bool ok = true;
        auto exchange = [&](int k, float2 v) -> float2 {
            float2* slot = xch + (k & 1) * 256;
            slot[hf * 128 + row] = v;
            mbar_arrive(&xbar[k * 4 + q4]);
            if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(&xbar[k * 4 + q4], 0, p.ctl, 90 + k));
            return slot[(1 - hf) * 128 + row];
        };
        if (p.fold) {
            // ---- q_hat and dA formed here from the raw tiles (one pass less over HBM than a separate
            // kernel): dA = dout * sigmoid(gate) in place over dout (gated layers), then
            // q_hat = RoPE(RMSNorm(q) * wq) in bf16 over the gate tile.  Each thread owns the 64
            // columns of its half row; the rotated pairs (j, j + half), half <= 32, lie in half 0.
            if (!__all_sync(0xffffffffu, mbar_wait(ld_full, 0, p.ctl, 108))) ok = false;
            uint8_t* qtile = smem + QP_Q;
            uint8_t* dtile = smem + QP_DA;
            const uint8_t* xtile = smem + QP_X;
            if (ok && gated) {
#pragma unroll 2
                for (int c8 = 8 * hf; c8 < 8 * hf + 8; ++c8) {
                    uint4* pd = reinterpret_cast<uint4*>(dtile + (c8 >> 3) * CH128 + sw128_off(row, c8 & 7));
                    const uint4 dd = *pd;
                    const uint4 go = ld_row8(qtile, row, c8);
                    const uint32_t dw[4] = {dd.x, dd.y, dd.z, dd.w}, gw[4] = {go.x, go.y, go.z, go.w};
                    uint32_t o[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2)  // the same arithmetic as the prep kernel's dA
                        o[k2] = pack_bf16x2(bf16lo(dw[k2]) * sigmoid_f32(bf16lo(gw[k2])),
                                            bf16hi(dw[k2]) * sigmoid_f32(bf16hi(gw[k2])));
                    *pd = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            float ssq = 0.f;
            if (ok) {
#pragma unroll 2
                for (int c8 = 8 * hf; c8 < 8 * hf + 8; ++c8) {
                    const uint4 u = ld_row8(xtile, row, c8);
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                        const float a = bf16lo(uw[k2]), c = bf16hi(uw[k2]);
                        ssq = fmaf(a, a, fmaf(c, c, ssq));
                    }
                }
            }
            ssq += exchange(7, make_float2(ssq, 0.f)).x;
            if (ok) {
                const float inv = ssq > 0.f || p.eps > 0.f ? rsqrtf(ssq * (1.0f / D) + p.eps) : 0.f;
                const int half = p.rope.half;
                const int c_first = hf == 0 ? (2 * half + 7) / 8 : 8;  // chunks [c_first, 8 hf + 8) are not rotated
                {
                    // the rotated pairs are split between the row's two threads (after the exchange above,
                    // both have read their gate columns, so either may write q_hat anywhere in half 0)
                    const int pos = valid_row && idx_ok(p.ctl, static_cast<long long>(b) * p.L + t,
                                                        static_cast<long long>(p.B) * p.L, 158)
                                        ? __ldg(p.pos + static_cast<long long>(b) * p.L + t)
                                        : 0;
                    const int j_mid = (half + 1) / 2;
#pragma unroll 1
                    for (int j = hf == 0 ? 0 : j_mid; j < (hf == 0 ? j_mid : half); ++j) {
                        const float a = ld_bf16(sw_elem(const_cast<uint8_t*>(xtile), CH128, row, j)) * inv * w_s[j];
                        const float c = ld_bf16(sw_elem(const_cast<uint8_t*>(xtile), CH128, row, j + half)) * inv * w_s[j + half];
                        float cs, sn;
                        rope_cos_sin(pos, p.rope.f_hi[j], p.rope.f_lo[j], cs, sn);
                        st_bf16(sw_elem(qtile, CH128, row, j), a * cs - c * sn);
                        st_bf16(sw_elem(qtile, CH128, row, j + half), c * cs + a * sn);
                    }
                }
                if (hf == 0) {
#pragma unroll 1
                    for (int e = 2 * half; e < 8 * c_first; ++e)
                        st_bf16(sw_elem(qtile, CH128, row, e), ld_bf16(sw_elem(const_cast<uint8_t*>(xtile), CH128, row, e)) * inv * w_s[e]);
                }
#pragma unroll 1
                for (int c8 = hf == 0 ? c_first : 8; c8 < 8 * hf + 8; ++c8) {
                    const uint4 u = ld_row8(xtile, row, c8);
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
                    const float* w = w_s + 8 * c8;
                    uint32_t o[4];
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2)
                        o[k2] = pack_bf16x2(bf16lo(uw[k2]) * inv * w[2 * k2], bf16hi(uw[k2]) * inv * w[2 * k2 + 1]);
                    *reinterpret_cast<uint4*>(qtile + (c8 >> 3) * CH128 + sw128_off(row, c8 & 7)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_async_smem();
            }
            tc_fence_before();
            mbar_arrive(qd_ready);
        }
        float m = 0.f, l = 0.f;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full, 0, p.ctl, 104));
        float mx = -INFINITY;
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < 5; ++k) {
                uint32_t r[16];
                tmem_ld16(lane_addr + C_S + c0 + 16 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = c0 + 16 * k + i;
                    if (c >= lo && c <= hi) mx = fmaxf(mx, __uint_as_float(r[i]));
                }
            }
        }
        mx = fmaxf(mx, exchange(0, make_float2(mx, 0.f)).x);
        m = (valid_row && mx > -INFINITY) ? mx * sl : 0.f;
        float lp = 0.f;
        if (ok) {
#pragma unroll 1
            for (int k = 0; k < 5; ++k) {
                uint32_t r[16], pk[8];
                tmem_ld16(lane_addr + C_S + c0 + 16 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const int c = c0 + 16 * k + i;
                    const bool v0 = valid_row && c >= lo && c <= hi, v1 = valid_row && c + 1 >= lo && c + 1 <= hi;
                    const float e0 = v0 ? ex2_approx(fmaf(__uint_as_float(r[i]), sl, -m)) : 0.f;
                    const float e1 = v1 ? ex2_approx(fmaf(__uint_as_float(r[i + 1]), sl, -m)) : 0.f;
                    pk[i / 2] = pack_bf16x2(e0, e1);
                    const float2 f = bf2f2(pk[i / 2]);  // the sum of the rounded values the MMA uses
                    lp += f.x + f.y;
                }
                tmem_st8(lane_addr + C_S + c0 + 8 * k, pk);  // P over S: these columns are already read
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_ready);
        l = lp + exchange(1, make_float2(lp, 0.f)).x;
        if (!ok) fail();
        const float il = l > 0.f ? 1.0f / l : 0.f;
        // ---- A = O / l on this warp's 64 columns, D = dA . A (pair sum), dgate
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(o_full, 0, p.ctl, 105));
        if (ok && gated && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(gd_full, 0, p.ctl, 108));
        float Dp = 0.f;
        uint8_t* dg_t = smem + (hf ? QP_DG1 : QP_DG0);
        if (ok) {
            tc_fence_after();
            const uint8_t* dout_t = smem + QP_DA;  // dout (gated: reloaded; ungated: dA is dout)
            const uint8_t* gate_t = smem + QP_Q;
#pragma unroll 1
            for (int k = 2 * hf; k < 2 * hf + 2; ++k) {
                uint32_t r[32];
                tmem_ld32(lane_addr + C_O + 32 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int v8 = 0; v8 < 4; ++v8) {
                    const uint4 du = ld_row8(dout_t, row, 4 * k + v8);
                    const uint32_t dw[4] = {du.x, du.y, du.z, du.w};
                    if (gated) {
                        const uint4 gu = ld_row8(gate_t, row, 4 * k + v8);
                        const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
                        float dg[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float gv = (e & 1) ? bf16hi(gw[e / 2]) : bf16lo(gw[e / 2]);
                            float sg, sgc;  // sigma and 1 - sigma, neither by subtraction
                            sigmoid_pair(gv, sg, sgc);
                            const float a = __uint_as_float(r[8 * v8 + e]) * il;
                            const float dav = ((e & 1) ? bf16hi(dw[e / 2]) : bf16lo(dw[e / 2])) * sg;
                            // D from the bf16 dA the dP product used (the prep kernel's rounding of
                            // the same value), so that sum_j dS_ij = 0 holds to fp32 rounding
                            Dp = fmaf(__bfloat162float(__float2bfloat16_rn(dav)), a, Dp);
                            dg[e] = dav * a * sgc;
                        }
                        // box k & 1 of this half's staging: row `row`, 16-byte chunks 2 v8, 2 v8 + 1
                        uint8_t* bx = dg_t + (k & 1) * (128 * 128) + row * 128;
                        *reinterpret_cast<float4*>(bx + (((2 * v8) ^ (row & 7)) << 4)) =
                            make_float4(dg[0], dg[1], dg[2], dg[3]);
                        *reinterpret_cast<float4*>(bx + (((2 * v8 + 1) ^ (row & 7)) << 4)) =
                            make_float4(dg[4], dg[5], dg[6], dg[7]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float a = __uint_as_float(r[8 * v8 + e]) * il;
                            Dp = fmaf((e & 1) ? bf16hi(dw[e / 2]) : bf16lo(dw[e / 2]), a, Dp);
                        }
                    }
                }
            }
        }
        if (gated) {
            fence_async_smem();
            mbar_arrive(&stg_full[hf]);
            if (q4 == 0 && lane == 0 && ok) {
                // rows past the sequence end fall outside the tensor and are not stored
                if (mbar_wait(&stg_full[hf], 0, p.ctl, 99)) {
                    tma_store_4d(&p.tm_dg, dg_t, 64 * hf, g * G, t0, b);
                    tma_store_4d(&p.tm_dg, dg_t + 128 * 128, 64 * hf + 32, g * G, t0, b);
                    bulk_commit();
                } else {
                    ok = false;
                }
            }
            ok = __all_sync(0xffffffffu, ok);
        }
        const float Dd = Dp + exchange(2, make_float2(Dp, 0.f)).x;
        if (ok && hf == 0 && valid_row && idx_ok(p.ctl, qrow, static_cast<long long>(p.B) * p.L * p.Hq, 152))
            p.stat[qrow] = make_float4(m, il, Dd, 0.f);
        // ---- dS = P (dP - D) / l on this warp's 80 keys, packed bf16 over dP
        if (ok) {
#pragma unroll 1
            for (int k = 0; k < 5; ++k) {
                uint32_t pr[8], r[16], d8[8];
                tmem_ld8(lane_addr + C_S + c0 + 8 * k, pr);
                tmem_ld16(lane_addr + C_DP + c0 + 16 * k, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 pp = bf2f2(pr[i]);
                    d8[i] = pack_bf16x2(pp.x * il * (__uint_as_float(r[2 * i]) - Dd),
                                        pp.y * il * (__uint_as_float(r[2 * i + 1]) - Dd));
                }
                tmem_st8(lane_addr + C_DP + c0 + 8 * k, d8);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(ds_ready);
        if (!ok) fail();
        // ---- dq: dQ_hat * c back through RoPE and RMSNorm, out by bulk tensor stores
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(dq_full, 0, p.ctl, 106));
        uint8_t* dq_t = smem + QP_DQ;  // every product is done: Q_hat, dA and K_hat are free
        float2* rope_tab = reinterpret_cast<float2*>(smem + QP_ROPE) + tt * kMaxRotHalf;
        if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int k = 2 * hf; k < 2 * hf + 2; ++k) {
                uint32_t v[32];
                tmem_ld32(lane_addr + C_O + 32 * k, v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *f32_chunk(dq_t, row, 8 * k + c) =
                        make_float4(__uint_as_float(v[4 * c]) * p.scale, __uint_as_float(v[4 * c + 1]) * p.scale,
                                    __uint_as_float(v[4 * c + 2]) * p.scale, __uint_as_float(v[4 * c + 3]) * p.scale);
            }
            // cos / sin of this row's token: its eight threads (4 rows x 2 halves) share the pairs
            const long long pi = static_cast<long long>(b) * p.L + t;
            const int pos = valid_row && idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 153) ? __ldg(p.pos + pi) : 0;
            for (int j = (row % G) * 2 + hf; j < p.rope.half; j += 2 * G) {
                float cs, sn;
                rope_cos_sin(pos, p.rope.f_hi[j], p.rope.f_lo[j], cs, sn);
                rope_tab[j] = make_float2(cs, sn);
            }
        }
        (void)exchange(3, make_float2(0.f, 0.f));  // both halves staged, the table is complete
        const int half = p.rope.half;
        if (ok && valid_row) {
            for (int j = hf; j < half; j += 2) {  // pairs split between the halves
                const float2 c = rope_tab[j];
                float* pa = f32_elem(dq_t, row, j);
                float* pb = f32_elem(dq_t, row, j + half);
                const float a = *pa, bb = *pb;
                *pa = a * c.x + bb * c.y;
                *pb = bb * c.x - a * c.y;
            }
        }
        (void)exchange(4, make_float2(0.f, 0.f));  // rotated
        float ss = 0.f, tw = 0.f;
        const uint8_t* xt = smem + QP_X;
        if (ok) {
#pragma unroll 4
            for (int c8 = 8 * hf; c8 < 8 * hf + 8; ++c8) {
                const uint4 u = ld_row8(xt, row, c8);
                const float4 y0 = *f32_chunk(dq_t, row, 2 * c8), y1 = *f32_chunk(dq_t, row, 2 * c8 + 1);
                const float x[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                                    bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
                const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ss = fmaf(x[e], x[e], ss);
                    tw = fmaf(x[e] * w_s[8 * c8 + e], y[e], tw);
                }
            }
        }
        const float2 other = exchange(5, make_float2(ss, tw));
        ss += other.x;
        tw += other.y;
        if (ok) {
            if (valid_row) {
                const float inv = ss > 0.f || p.eps > 0.f ? rsqrtf(ss * (1.0f / D) + p.eps) : 0.f;
                const float coef = inv * inv * inv * tw * (1.0f / D);
#pragma unroll 4
                for (int c8 = 8 * hf; c8 < 8 * hf + 8; ++c8) {
                    const uint4 u = ld_row8(xt, row, c8);
                    float4* p0 = f32_chunk(dq_t, row, 2 * c8);
                    float4* p1 = f32_chunk(dq_t, row, 2 * c8 + 1);
                    const float4 y0 = *p0, y1 = *p1;
                    const float* w = w_s + 8 * c8;
                    *p0 = make_float4(inv * w[0] * y0.x - coef * bf16lo(u.x), inv * w[1] * y0.y - coef * bf16hi(u.x),
                                      inv * w[2] * y0.z - coef * bf16lo(u.y), inv * w[3] * y0.w - coef * bf16hi(u.y));
                    *p1 = make_float4(inv * w[4] * y1.x - coef * bf16lo(u.z), inv * w[5] * y1.y - coef * bf16hi(u.z),
                                      inv * w[6] * y1.z - coef * bf16lo(u.w), inv * w[7] * y1.w - coef * bf16hi(u.w));
                }
            }
            fence_async_smem();
        }
        mbar_arrive(dq_stg);
        if (threadIdx.x == 0 && ok) {
            if (mbar_wait(dq_stg, 0, p.ctl, 98)) {
                for (int k = 0; k < 4; ++k) tma_store_4d(&p.tm_dqf, dq_t + k * F32BOX, 32 * k, g * G, t0, b);
                bulk_commit();
            } else {
                ok = false;
            }
        }
        if (q4 == 0 && lane == 0) bulk_wait_all();  // this half's dgate stores (and dq) have landed
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
    if (warp == 8) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------- kernel 3: key pass
constexpr int kKThreads = 288;  // warps 0-7 rows (two column halves), warp 8 TMA + MMA

__global__ void __launch_bounds__(kKThreads, 1) bwd_kpass_kernel(const __grid_constant__ BackwardTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + KP_BAR);
    uint64_t* kv_full = bar + 0;
    uint64_t* qd_full = bar + 1;   // [2] ring stage
    uint64_t* qd_empty = bar + 3;  // [2] ring stage
    uint64_t* s_full = bar + 5;    // [2] column half
    uint64_t* p_ready = bar + 7;   // [2] column half
    uint64_t* done = bar + 9;
    uint64_t* x_full = bar + 10;   // raw k tile
    uint64_t* dv_stg = bar + 11;   // dv staging written (128 arrivals)
    uint64_t* dk_stg = bar + 12;   // dk staging written (128 arrivals)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + KP_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + KP_MISC + 4);
    float* w_s = reinterpret_cast<float*>(smem + KP_W);
    float4* stat_s = reinterpret_cast<float4*>(smem + KP_STAT);  // [8 warps][64]
    // TMEM: S^T [0, 128) and dP^T [128, 256), each as two 64-column halves (one per half of
    // the query tile; P^T / dS^T of a half are packed into the first 32 columns of that half),
    // dV [256, 384), dK_hat [384, 512)
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
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 128);
        }
        mbar_init(done, 1);
        mbar_init(x_full, 1);
        mbar_init(dv_stg, 128);
        mbar_init(dk_stg, 128);
        fence_barrier_init();
    }
    if (threadIdx.x < 32)
        *reinterpret_cast<float4*>(w_s + lane * 4) = __ldg(reinterpret_cast<const float4*>(p.wk + lane * 4));
    if (warp == 8) {
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

    if (warp == 8) {
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_qh);
            tma_prefetch_desc(&p.tm_da);
            tma_prefetch_desc(&p.tm_kk);
            tma_prefetch_desc(&p.tm_vk);
            tma_prefetch_desc(&p.tm_kraw);
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
            constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false, false);
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, false, true);
            auto issue_s = [&](int n, int h) {  // S^T and dP^T of the query rows [64 h, 64 h + 64) of tile n
                const uint32_t qd = KP_QD + (n & 1) * 2 * TILE128 + h * 64 * 128;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_S + 64 * h, sdesc(sbase + KP_K + co, 16, 1024, kSw128),
                              sdesc(sbase + qd + co, 16, 1024, kSw128), id_s, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_DP + 64 * h, sdesc(sbase + KP_V + co, 16, 1024, kSw128),
                              sdesc(sbase + qd + TILE128 + co, 16, 1024, kSw128), id_s, ks > 0);
                }
                umma_commit(&s_full[h]);
            };
            auto issue_acc = [&](int n, int h) {  // dV += P^T dA, dK_hat += dS^T Q_hat over those rows
                const uint32_t qd = KP_QD + (n & 1) * 2 * TILE128 + h * 64 * 128;
#pragma unroll
                for (int ks = 0; ks < 64 / 16; ++ks) {
                    const uint32_t acc = (n > 0 || h > 0 || ks > 0) ? 1u : 0u;
                    umma_tmem_a(tbase + C_DV, tbase + C_S + 64 * h + ks * 8,
                                sdesc(sbase + qd + TILE128 + ks * 16 * 128, CH128, 1024, kSw128), id_o, acc);
                    umma_tmem_a(tbase + C_DK, tbase + C_DP + 64 * h + ks * 8,
                                sdesc(sbase + qd + ks * 16 * 128, CH128, 1024, kSw128), id_o, acc);
                }
            };
            load_qd(0);
            if (n_tiles > 1) load_qd(1);
            bool ok = mbar_wait(kv_full, 0, p.ctl, 111) && mbar_wait(&qd_full[0], 0, p.ctl, 112);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(0, 1);
            }
            // per tile: half 0's accumulation, then (once the next tile is in) the next
            // tile's half-0 scores, so the warps of half 0 move on while half 1 finishes
            for (int n = 0; n < n_tiles && ok && !aborted(); ++n) {
                const bool more = n + 1 < n_tiles;
                ok = mbar_wait(&p_ready[0], n & 1, p.ctl, 113);
                if (!ok) break;
                tc_fence_after();
                issue_acc(n, 0);
                if (more) {
                    ok = mbar_wait(&qd_full[(n + 1) & 1], ((n + 1) >> 1) & 1, p.ctl, 114);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(n + 1, 0);
                }
                ok = mbar_wait(&p_ready[1], n & 1, p.ctl, 120);
                if (!ok) break;
                tc_fence_after();
                issue_acc(n, 1);
                umma_commit(&qd_empty[n & 1]);
                if (more) issue_s(n + 1, 1);
                if (n + 2 < n_tiles) {
                    ok = mbar_wait(&qd_empty[n & 1], (n >> 1) & 1, p.ctl, 115);
                    if (!ok) break;
                    load_qd(n + 2);
                }
            }
            umma_commit(done);
            // the raw keys for the RMSNorm backward, into the ring once every product is done
            if (ok) ok = mbar_wait(done, 0, p.ctl, 118);
            if (ok) {
                mbar_arrive_expect_tx(x_full, TILE128);
                for (int ch = 0; ch < 2; ++ch)
                    tma_load_4d(smem + KP_X + ch * CH128, &p.tm_kraw, x_full, ch * 64, g, j0, b);
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ rows (thread = key row = TMEM lane;
        // warps 0-3 the query columns [0, 64) of every tile, warps 4-7 the columns [64, 128))
        const int h = warp >> 2;
        const int row = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int kj = j0 + row;
        const bool valid_key = kj < p.L;
        const float sl = p.scale_log2;
        const int W = p.window;
        bool ok = true;
        for (int n = 0; n < n_tiles && ok; ++n) {
            const int u0 = j0 + n * T;
            // the statistics of this half's 64 query rows, one copy per warp (no barrier across
            // warps: a warp that gives up on a wait must not leave the others blocked)
            float4* sts = stat_s + warp * 64;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int c = 64 * h + lane + 32 * i;
                const int u = u0 + c / G;
                const long long si = (static_cast<long long>(b) * p.L + u) * p.Hq + g * G + c % G;
                sts[lane + 32 * i] = u < p.L && idx_ok(p.ctl, si, static_cast<long long>(p.B) * p.L * p.Hq, 154)
                                         ? p.stat[si]
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncwarp();
            if (aborted() || !__all_sync(0xffffffffu, mbar_wait(&s_full[h], n & 1, p.ctl, 116))) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                uint32_t r[32], dp[32], pp[16], dd[16];
                tmem_ld32(lane_addr + C_S + 64 * h + 32 * k, r);
                tmem_ld32(lane_addr + C_DP + 64 * h + 32 * k, dp);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float pv[2], dv2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int cl = 32 * k + i + e;  // column within the half
                        const int u = u0 + (64 * h + cl) / G;
                        const float4 s4 = sts[cl];
                        const bool v = valid_key && u >= kj && u - kj < W && u < p.L;
                        const float pr = v ? ex2_approx(fmaf(__uint_as_float(r[i + e]), sl, -s4.x)) * s4.y : 0.f;
                        pv[e] = pr;
                        dv2[e] = pr * (__uint_as_float(dp[i + e]) - s4.z);
                    }
                    pp[i / 2] = pack_bf16x2(pv[0], pv[1]);
                    dd[i / 2] = pack_bf16x2(dv2[0], dv2[1]);
                }
                tmem_st16(lane_addr + C_S + 64 * h + 16 * k, pp);   // P^T over S^T (columns already read)
                tmem_st16(lane_addr + C_DP + 64 * h + 16 * k, dd);  // dS^T over dP^T
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_ready[h]);
        }
        if (!ok) fail();
        if (warp < 4) {
            // ---- epilogue (warps 0-3): dV, then dK_hat back through RoPE and RMSNorm; both leave
            // by bulk tensor stores (rows past the sequence end fall outside the tensor)
            if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(done, 0, p.ctl, 117));
            uint8_t* dv_t = smem + KP_DV;
            uint8_t* dk_t = smem + KP_DK;
            if (ok) {
                tc_fence_after();
                tmem_row_to_tile(lane_addr + C_DV, dv_t, row, 1.0f);
                fence_async_smem();
            }
            mbar_arrive(dv_stg);
            if (row == 0 && ok) {
                if (mbar_wait(dv_stg, 0, p.ctl, 97)) {
                    for (int k = 0; k < 4; ++k) tma_store_4d(&p.tm_dvf, dv_t + k * F32BOX, 32 * k, g, j0, b);
                    bulk_commit();
                } else {
                    ok = false;
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tmem_row_to_tile(lane_addr + C_DK, dk_t, row, p.scale);
                if (!aborted()) ok = __all_sync(0xffffffffu, mbar_wait(x_full, 0, p.ctl, 119));
            }
            if (ok) {
                if (valid_key) {
                    const long long pi = static_cast<long long>(b) * p.L + kj;
                    const int pos = idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 155) ? __ldg(p.pos + pi) : 0;
                    row_norm_rope_bwd(dk_t, row, smem + KP_X, w_s, p.eps, p.rope.half, [&](int j) {
                        float cs, sn;
                        rope_cos_sin(pos, p.rope.f_hi[j], p.rope.f_lo[j], cs, sn);
                        return make_float2(cs, sn);
                    });
                }
                fence_async_smem();
            }
            mbar_arrive(dk_stg);
            if (row == 0 && ok) {
                if (mbar_wait(dk_stg, 0, p.ctl, 96)) {
                    for (int k = 0; k < 4; ++k) tma_store_4d(&p.tm_dkf, dk_t + k * F32BOX, 32 * k, g, j0, b);
                    bulk_commit();
                } else {
                    ok = false;
                }
            }
            if (row == 0) bulk_wait_all();
            if (!ok) fail();
        }
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        const long long c0 = clock64();
        while (clock64() - c0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 8) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------- global layer: query pass
// The global layer (every earlier key, no gate): the query tile of 32 tokens x 4 heads sees
// the keys [0, t0 + 32), in blocks of 128, so its row statistics need every block first.
//   loop 1, per block: S = Q_hat K_hat^T and dP = dA V^T into TMEM; each row keeps, per column
//     half, a running maximum m (log2-scaled scores), l = sum of 2^(s c log2e - m) and
//     D' = sum of the same weights times dP, rescaled when m moves; the halves merge into
//     (m, 1 / l, D = D' / l) with D = rowsum(P dP) = rowsum(dA A), which go to the workspace in
//     the windowed pass's format, for the key pass (run with window = L).
//   loop 2, per block: S and dP again, P from the statistics, dS = P (dP - D) packed bf16 over
//     dP, dQ_hat += dS K_hat in TMEM.
//   dQ_hat then goes back through RoPE and RMSNorm into dq (fp32), as in the windowed pass.
// Warps 0-7: rows (thread = row = TMEM lane; warp w has the lane quarter w & 3 and the column
// half w >> 2 of every key block); warp 8: TMA (one thread); warp 9: MMA (one thread), TMEM.
constexpr int kGThreads = 320;
constexpr uint32_t GQ_Q = 0;                        // Q_hat tile
constexpr uint32_t GQ_DA = GQ_Q + TILE128;          // dA tile
constexpr uint32_t GQ_RING = GQ_DA + TILE128;       // 2 stages x (K_hat block, V block)
constexpr uint32_t GQ_XCH = GQ_RING + 4 * TILE128;  // [2 halves][128 rows] float4 (m, l, D', 0)
constexpr uint32_t GQ_W = GQ_XCH + 2 * 128 * 16;    // wq [D]
constexpr uint32_t GQ_BAR = GQ_W + D * 4;
constexpr uint32_t GQ_MISC = GQ_BAR + 16 * 8;
constexpr uint32_t GQ_SMEM = GQ_MISC + 32;
constexpr uint32_t GQ_DQ = GQ_RING;                 // dq staging (four fp32 boxes), ring free at the end
constexpr uint32_t GQ_X = GQ_RING + 2 * TILE128;    // raw q tile, loaded into the free ring at the end
static_assert(GQ_DQ + F32TILE <= GQ_X && GQ_X + TILE128 <= GQ_XCH, "staging inside the ring");
static_assert(GQ_RING % 1024 == 0 && GQ_X % 1024 == 0, "swizzle atoms");
static_assert(GQ_SMEM <= 227 * 1024, "shared memory");

__global__ void __launch_bounds__(kGThreads, 1) bwd_qpass_global_kernel(const __grid_constant__ BackwardTcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + GQ_BAR);
    uint64_t* q_full = bar + 0;
    uint64_t* kv_full = bar + 1;   // [2]
    uint64_t* kv_empty = bar + 3;  // [2]
    uint64_t* s_full = bar + 5;
    uint64_t* s_free = bar + 6;    // loop 1: the rows have S and dP in registers (256 arrivals)
    uint64_t* ds_ready = bar + 7;  // loop 2: dS is in TMEM (256 arrivals)
    uint64_t* dq_full = bar + 8;
    uint64_t* x_full = bar + 9;
    uint64_t* st_xch = bar + 10;   // both halves' statistics are in shared memory (256 arrivals)
    uint64_t* dq_stg = bar + 11;   // dq staging written (128 arrivals)
    uint64_t* dq_done = bar + 12;  // loop 2: the dQ product of a block has read its dS
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + GQ_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + GQ_MISC + 4);
    float* w_s = reinterpret_cast<float*>(smem + GQ_W);
    float4* xch = reinterpret_cast<float4*>(smem + GQ_XCH);
    // TMEM: S, dP, dQ_hat (fp32, 128 columns each) and dS (bf16 packed, 64 columns: half h's keys in
    // columns [32 h, 32 h + 32)), so the next block's S and dP products run while dS is formed
    constexpr uint32_t C_S = 0, C_DP = 128, C_DQ = 256, C_DS = 384;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbg = p.B * p.Hkv;
    const int n_qt = (p.L + T - 1) / T;
    const int t0 = (n_qt - 1 - static_cast<int>(blockIdx.x / nbg)) * T;  // heaviest (most key blocks) first
    const int g = static_cast<int>(blockIdx.x % nbg) % p.Hkv;
    const int b = static_cast<int>(blockIdx.x % nbg) / p.Hkv;
    const int nblk = (t0 + T + BK - 1) / BK;  // key blocks [0, nblk), each visited by both loops

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 130, kErrAlign);
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 256);
        mbar_init(ds_ready, 256);
        mbar_init(dq_full, 1);
        mbar_init(x_full, 1);
        mbar_init(st_xch, 256);
        mbar_init(dq_stg, 128);
        mbar_init(dq_done, 1);
        fence_barrier_init();
    }
    if (threadIdx.x < 32)
        *reinterpret_cast<float4*>(w_s + lane * 4) = __ldg(reinterpret_cast<const float4*>(p.wq + lane * 4));
    if (warp == 9) {
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

    if (warp == 8) {
        // ------------------------------------------------------------ TMA
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_qh);
            tma_prefetch_desc(&p.tm_da);
            tma_prefetch_desc(&p.tm_kk);
            tma_prefetch_desc(&p.tm_vk);
            tma_prefetch_desc(&p.tm_q);
            mbar_arrive_expect_tx(q_full, 2 * TILE128);
            for (int ch = 0; ch < 2; ++ch) {
                tma_load_4d(smem + GQ_Q + ch * CH128, &p.tm_qh, q_full, ch * 64, g * G, t0, b);
                tma_load_4d(smem + GQ_DA + ch * CH128, &p.tm_da, q_full, ch * 64, g * G, t0, b);
            }
            bool ok = true;
            for (int n = 0; n < 2 * nblk && ok && !aborted(); ++n) {  // loop 1 then loop 2: blocks n mod nblk
                const int st = n & 1, j = n % nblk;
                ok = mbar_wait(&kv_empty[st], ((n >> 1) & 1) ^ 1, p.ctl, 131);
                if (!ok) break;
                uint8_t* dst = smem + GQ_RING + st * 2 * TILE128;
                mbar_arrive_expect_tx(&kv_full[st], 2 * TILE128);
                for (int ch = 0; ch < 2; ++ch) {
                    tma_load_4d(dst + ch * CH128, &p.tm_kk, &kv_full[st], ch * 64, g, j * BK, b);
                    tma_load_4d(dst + TILE128 + ch * CH128, &p.tm_vk, &kv_full[st], ch * 64, g, j * BK, b);
                }
            }
            // the raw q rows for the RMSNorm backward, into the ring once every product is done
            if (ok) ok = mbar_wait(dq_full, 0, p.ctl, 132);
            if (ok) {
                mbar_arrive_expect_tx(x_full, TILE128);
                for (int ch = 0; ch < 2; ++ch)
                    tma_load_4d(smem + GQ_X + ch * CH128, &p.tm_q, x_full, ch * 64, g * G, t0, b);
            }
            if (!ok) fail();
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA
        if (lane == 0 && !aborted()) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, BK, false, false);  // S, dP: both operands K-major
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, false, true);    // dQ: K_hat block MN-major
            bool ok = mbar_wait(q_full, 0, p.ctl, 133);
            // dQ_hat += dS K_hat for loop-2 block m (its K_hat in stage st_m)
            auto issue_dq = [&](int m, int st_m) {
                const uint32_t kofs = GQ_RING + st_m * 2 * TILE128;
#pragma unroll
                for (int ks = 0; ks < BK / 16; ++ks)
                    umma_tmem_a(tbase + C_DQ, tbase + C_DS + 32 * (ks >> 2) + 8 * (ks & 3),
                                sdesc(sbase + kofs + ks * 16 * 128, CH128, 1024, kSw128), id_o,
                                (m > 0 || ks > 0) ? 1u : 0u);
                umma_commit(dq_done);
                umma_commit(&kv_empty[st_m]);
            };
            for (int n = 0; n < 2 * nblk && ok && !aborted(); ++n) {
                const int st = n & 1;
                const uint32_t kofs = GQ_RING + st * 2 * TILE128, vofs = kofs + TILE128;
                ok = mbar_wait(&kv_full[st], (n >> 1) & 1, p.ctl, 134);
                // S and dP of the previous block must be in the rows' registers
                if (ok && n > 0) ok = mbar_wait(s_free, (n - 1) & 1, p.ctl, 135);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_S, sdesc(sbase + GQ_Q + co, 16, 1024, kSw128),
                              sdesc(sbase + kofs + co, 16, 1024, kSw128), id_s, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t co = (ks >> 2) * CH128 + (ks & 3) * 32;
                    umma_bf16(tbase + C_DP, sdesc(sbase + GQ_DA + co, 16, 1024, kSw128),
                              sdesc(sbase + vofs + co, 16, 1024, kSw128), id_s, ks > 0);
                }
                umma_commit(s_full);
                if (n < nblk) {
                    umma_commit(&kv_empty[st]);
                    continue;
                }
                // loop 2: the previous block's dQ once its dS is in TMEM (this block's S / dP run meanwhile)
                const int m = n - nblk;
                if (m > 0) {
                    ok = mbar_wait(ds_ready, (m - 1) & 1, p.ctl, 136);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dq(m - 1, (n - 1) & 1);
                }
            }
            if (ok && !aborted()) {  // the last block's dQ
                ok = mbar_wait(ds_ready, (nblk - 1) & 1, p.ctl, 143);
                if (ok) {
                    tc_fence_after();
                    issue_dq(nblk - 1, (2 * nblk - 1) & 1);
                }
            }
            umma_commit(dq_full);
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ rows
        const int q4 = warp & 3, hf = warp >> 2;
        const int row = q4 * 32 + lane;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>(q4 * 32) << 16);
        const int t = t0 + row / G;
        const bool valid_row = t < p.L;
        const float sl = p.scale_log2;
        float m = -INFINITY, l = 0.f, dsum = 0.f;  // this half's running max, weight sum, D'
        bool ok = true;
        auto load_block = [&](uint32_t (&s)[64], uint32_t (&dp)[64]) {
            tmem_ld32(lane_addr + C_S + 64 * hf, s);
            tmem_ld32(lane_addr + C_S + 64 * hf + 32, s + 32);
            tmem_ld32(lane_addr + C_DP + 64 * hf, dp);
            tmem_ld32(lane_addr + C_DP + 64 * hf + 32, dp + 32);
            tmem_wait_ld();
        };
        for (int n = 0; n < nblk && ok; ++n) {
            if (aborted() || !__all_sync(0xffffffffu, mbar_wait(s_full, n & 1, p.ctl, 137))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[64], dp[64];
            load_block(s, dp);
            tc_fence_before();
            mbar_arrive(s_free);
            const int kmax = t - (n * BK + 64 * hf);  // columns c <= kmax hold keys <= t
            float bm = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c)
                if (c <= kmax) bm = fmaxf(bm, __uint_as_float(s[c]));
            const float m_new = fmaxf(m, bm * sl);
            if (m_new != -INFINITY) {
                const float corr = ex2_approx(m - m_new);  // 0 while m is still -inf
                float ls = 0.f, dl = 0.f;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float e = c <= kmax ? ex2_approx(fmaf(__uint_as_float(s[c]), sl, -m_new)) : 0.f;
                    ls += e;
                    dl = fmaf(e, __uint_as_float(dp[c]), dl);
                }
                l = fmaf(l, corr, ls);
                dsum = fmaf(dsum, corr, dl);
                m = m_new;
            }
        }
        // merge the two column halves of every row
        xch[hf * 128 + row] = make_float4(m, l, dsum, 0.f);
        mbar_arrive(st_xch);
        if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(st_xch, 0, p.ctl, 138));
        const float4 o = xch[(1 - hf) * 128 + row];
        float mm = fmaxf(m, o.x), lt = 0.f, dt = 0.f;
        if (mm != -INFINITY) {
            const float c0 = ex2_approx(m - mm), c1 = ex2_approx(o.x - mm);
            lt = l * c0 + o.y * c1;
            dt = dsum * c0 + o.z * c1;
        } else {
            mm = 0.f;
        }
        const float inv_l = lt > 0.f ? 1.0f / lt : 0.f;
        const float dd = dt * inv_l;
        const long long si = (static_cast<long long>(b) * p.L + t) * p.Hq + g * G + row % G;
        if (hf == 0 && valid_row && ok && idx_ok(p.ctl, si, static_cast<long long>(p.B) * p.L * p.Hq, 156))
            p.stat[si] = make_float4(mm, inv_l, dd, 0.f);
        for (int n = 0; n < nblk && ok; ++n) {
            if (aborted() || !__all_sync(0xffffffffu, mbar_wait(s_full, (nblk + n) & 1, p.ctl, 139))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[64], dp[64];
            load_block(s, dp);
            tc_fence_before();
            mbar_arrive(s_free);
            const int kmax = t - (n * BK + 64 * hf);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                float ds2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pr = c + e <= kmax
                                         ? ex2_approx(fmaf(__uint_as_float(s[c + e]), sl, -mm)) * inv_l
                                         : 0.f;
                    ds2[e] = pr * (__uint_as_float(dp[c + e]) - dd);
                }
                pk[c / 2] = pack_bf16x2(ds2[0], ds2[1]);
            }
            // the dS columns are free once the previous block's dQ product has read them
            if (n > 0 && (aborted() || !__all_sync(0xffffffffu, mbar_wait(dq_done, (n - 1) & 1, p.ctl, 144)))) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st16(lane_addr + C_DS + 32 * hf, pk);
            tmem_st16(lane_addr + C_DS + 32 * hf + 16, pk + 16);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(ds_ready);
        }
        if (!ok) fail();
        if (hf == 0) {
            // ---- epilogue (warps 0-3, thread = row): dQ_hat back through RoPE and RMSNorm into dq
            if (ok && !aborted()) ok = __all_sync(0xffffffffu, mbar_wait(dq_full, 0, p.ctl, 140));
            uint8_t* dq_t = smem + GQ_DQ;
            if (ok) {
                tc_fence_after();
                tmem_row_to_tile(lane_addr + C_DQ, dq_t, row, p.scale);
                if (!aborted()) ok = __all_sync(0xffffffffu, mbar_wait(x_full, 0, p.ctl, 141));
            }
            if (ok) {
                if (valid_row) {
                    const long long pi = static_cast<long long>(b) * p.L + t;
                    const int pos = idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 157) ? __ldg(p.pos + pi) : 0;
                    row_norm_rope_bwd(dq_t, row, smem + GQ_X, w_s, p.eps, p.rope.half, [&](int j) {
                        float cs, sn;
                        rope_cos_sin(pos, p.rope.f_hi[j], p.rope.f_lo[j], cs, sn);
                        return make_float2(cs, sn);
                    });
                }
                fence_async_smem();
            }
            mbar_arrive(dq_stg);
            if (row == 0 && ok) {
                if (mbar_wait(dq_stg, 0, p.ctl, 142)) {
                    for (int k = 0; k < 4; ++k) tma_store_4d(&p.tm_dqf, dq_t + k * F32BOX, 32 * k, g * G, t0, b);
                    bulk_commit();
                    bulk_wait_all();
                } else {
                    ok = false;
                }
            }
            if (!ok) fail();
        }
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        const long long c0 = clock64();
        while (clock64() - c0 < 4000000ll) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 9) tmem_dealloc(tbase, 512);
}

}  // namespace

bool backward_tc_supports(int d, int Hq, int Hkv, int window) {
    return d == D && Hkv > 0 && Hq == G * Hkv && window >= 1 && window <= 128;
}
bool backward_tc_global_supports(int d, int Hq, int Hkv) { return d == D && Hkv > 0 && Hq == G * Hkv; }

size_t backward_tc_workspace_bytes(int B, int L, int Hq, int Hkv) {
    const size_t rq = static_cast<size_t>(B) * L * Hq, rk = static_cast<size_t>(B) * L * Hkv;
    return rq * D * 2 * 2 + rk * D * 2 + rq * 16;  // q_hat, dA, k_hat (bf16), statistics
}

cudaError_t launch_backward_tc(const BackwardTcParams& p, cudaStream_t s) {
    const long long nq = static_cast<long long>(p.B) * p.L * p.Hq, nk = static_cast<long long>(p.B) * p.L * p.Hkv;
    if (nq == 0) return cudaSuccess;
    if (nq + nk >= (1ll << 31)) return cudaErrorInvalidValue;  // the prep kernel indexes rows in 32 bits
    BackwardTcParams pp = p;
    pp.prep_first = p.fold ? static_cast<int>(nq) : 0;  // fold: the query pass forms q_hat and dA, prep k_hat only
    const long long prep_rows = nq + nk - pp.prep_first;
    bwd_tc_prep_kernel<<<static_cast<unsigned>((prep_rows + 8 * kPrepRows - 1) / (8 * kPrepRows)), 256, 0, s>>>(pp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_kpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KP_SMEM);
    if (e != cudaSuccess) return e;
    const long long nbg = static_cast<long long>(p.B) * p.Hkv;
    if (p.global) {  // every earlier key: statistics over all key blocks, then dq; the key pass with window = L
        e = cudaFuncSetAttribute(bwd_qpass_global_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GQ_SMEM);
        if (e != cudaSuccess) return e;
        bwd_qpass_global_kernel<<<static_cast<unsigned>(nbg * ((p.L + T - 1) / T)), kGThreads, GQ_SMEM, s>>>(p);
    } else {
        e = cudaFuncSetAttribute(bwd_qpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QP_SMEM);
        if (e != cudaSuccess) return e;
        bwd_qpass_kernel<<<static_cast<unsigned>(nbg * ((p.L + T - 1) / T)), kQThreads, QP_SMEM, s>>>(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_kpass_kernel<<<static_cast<unsigned>(nbg * ((p.L + BK - 1) / BK)), kKThreads, KP_SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace zg
