// swa2_prefill.cu -- gated sliding-window GQA prefill, persistent warp-specialised
// kernel for GQA ratios G = Hq/Hkv in {2, 4, 8}.
//
// Computes what swa_prefill.cu documents ("ZGCM-1-7B 完全解説", gotosocial
// explainer, section "アーキテクチャ"; "ZGCM-1: A Fully Open and Extremely
// Efficient Foundation Model for Math and Agentic Search", jaehun.me review,
// section "게이트형 SWA의 동작"):  out_i = softmax_{j in [max(0,i-W+1), i]}
// (q_hat_i . k_hat_j / sqrt(d)) v_j * sigmoid(g_i), q_hat / k_hat after QK RMSNorm
// and partial RoPE.
//
// One CTA per SM walks a contiguous run of 128-row tiles (T = 128/G tokens x G
// query heads of one KV head).  Along a run the keys are shared: tile n needs
// the 128 keys before it plus its own T, i.e. the last NS = 128/T + 1 key slots
// of T keys.  Keys and values therefore live in a ring of NS + 1 slots in shared
// memory and each key is loaded and normalised once per run.
//
// Warp roles (20 warps):
//   warp 0      TMA loop (one thread): K slots into the key ring (refilled once the
//               last QK reading a slot has completed), V slots (after the last PV),
//               Q tiles into a 4-deep buffer ring, output stores.
//   warp 1      MMA loop (one thread), QK and PV as soon as each is ready (below).
//               Warp 1 owns TMEM (512 columns).
//   warps 4-11  RMSNorm + RoPE of the Q tile rows, in place (bf16 -> fp16), two
//               lanes per row, cos/sin shared by the lanes of one token.  The MMA
//               loop then issues S = Q K^T (fp16, M128 x N=NK, split in two when
//               the window wraps around the key ring) into one of two TMEM S buffers.
//   warps 2-3   the same for the K rows of every new slot.
//   warps 12-15 softmax: exp2 against a bound on the scores, bf16 P written back
//               over S in TMEM and the row sums l of that very bf16 P written to
//               TMEM, after which the MMA loop issues O = P V (P read from TMEM, V
//               MN-major from the ring); the softmax also fetches the gate tile into
//               the freed Q buffer.
//   warps 16-19 epilogue: O / l * sigmoid(gate), in place over the gate tile, which
//               the TMA loop then stores.
// Every hand-off is an mbarrier with a bounded wait; a wait that gives up sets
// the CTA's abort flag and every role winds down.
#include "zg_qk.cuh"

namespace zg {
namespace {

template <int D, int G>
struct Swa2 {
    static constexpr int T = 128 / G;         // tokens per tile
    static constexpr int WS = 128 / T;        // history slots (128 keys before the tile)
    static constexpr int NS = WS + 1;         // slots per tile window
    static constexpr int NK = NS * T;         // keys per tile (N of the QK product)
    static constexpr int SLOT2 = T * 128 * (D / 64) * 2;  // bytes of one K slot + one V slot
    static constexpr int NQB = 4;             // Q / gate / out buffers (4 measured 5% faster than 3)
    static constexpr int BASE_SMEM = NQB * 128 * 128 * (D / 64) + 2048 + 2 * D * 4;
    static constexpr int SPARE = (232448 - BASE_SMEM) / SLOT2 - (NS + 1);
    static constexpr int R = NS + 1 + (SPARE > 3 ? 3 : SPARE);  // ring slots
    static constexpr int RR = R * T;          // ring rows
    static constexpr int NCH = D / 64;        // 64-element chunks per head row
    static constexpr uint32_t QCH = 128 * 128;
    static constexpr uint32_t QBUF = QCH * NCH;
    static constexpr uint32_t KCH = RR * 128;
    static constexpr uint32_t RING = KCH * NCH;
    static constexpr uint32_t SLOT_BYTES = T * 128 * NCH;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + NQB * QBUF;
    static constexpr uint32_t OFF_V = OFF_K + RING;
    static constexpr uint32_t OFF_BAR = OFF_V + RING;
    static constexpr int NBAR = 4 * NQB + 5 * R + 2 * 3 + 2 + 3;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_W = (OFF_MISC + 16 + 15) / 16 * 16;  // wq [D], wk [D] fp32
    static constexpr uint32_t OFF_R = OFF_W + 2 * D * 4;  // rotation frequencies: f_hi [64], f_lo [64] fp32
    static constexpr uint32_t SMEM = OFF_R + 2 * kMaxRotHalf * 4;
    static constexpr int SCOLS = (NK + 31) / 32 * 32;  // TMEM columns of one S buffer
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int O_COL = 2 * SCOLS;
    static constexpr int L_COL = O_COL + D;  // 4 x 8 columns: row sums of P of tiles n mod 4
    static_assert(L_COL + 32 <= 512, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(T % 16 == 0 && NK <= 256, "tile shape");
};

constexpr int kThreads = 640;  // 20 warps

struct TileIdx {
    int b, g, lt;
};
__device__ __forceinline__ TileIdx decode_tile(long long idx, int n_lt, int Hkv) {
    TileIdx t;
    t.lt = static_cast<int>(idx % n_lt);
    const long long bg = idx / n_lt;
    t.g = static_cast<int>(bg % Hkv);
    t.b = static_cast<int>(bg / Hkv);
    return t;
}
// next tile in (b, g, lt) order, lt fastest (no division in the loops)
__device__ __forceinline__ void next_tile(TileIdx& t, int n_lt, int Hkv) {
    if (++t.lt == n_lt) {
        t.lt = 0;
        if (++t.g == Hkv) {
            t.g = 0;
            ++t.b;
        }
    }
}

// Walks the K/V slot stream of a CTA: at the start of a span (first tile of the run,
// or a sequence start) the WS history slots come first, then one slot per tile.
struct SlotCursor {
    TileIdx ti;
    int it, w, c;
    __device__ __forceinline__ void init(const TileIdx& first, int WS) {
        ti = first;
        it = 0;
        c = 0;
        w = WS;  // the run's first tile always starts a span
    }
    __device__ __forceinline__ int slot_tile() const { return ti.lt - w; }
    __device__ __forceinline__ void advance(int n_tiles, int n_lt, int Hkv, int WS) {
        ++c;
        if (w > 0) {
            --w;
            return;
        }
        ++it;
        if (it < n_tiles) {
            next_tile(ti, n_lt, Hkv);
            w = ti.lt == 0 ? WS : 0;
        }
    }
};

// ROT: rotary width compiled in (the dims then stay in registers), or 0 = any width.
// PRE: the inputs arrive pre-normalised (q_hat, k_hat in fp16, the gate as sigmoid(g) in bf16, as
// the fused projections of the whole layer write them): the Q / K transforms and the sigmoid are
// skipped and the tiles go to the tensor cores as loaded.
template <int D, int G, int ROT, bool PRE>
__global__ void __launch_bounds__(kThreads, 1) swa2_kernel(const __grid_constant__ PrefillParams p) {
    using C = Swa2<D, G>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bar;
    uint64_t* q_ready = q_full + C::NQB;
    uint64_t* g_full = q_ready + C::NQB;
    uint64_t* k_full = g_full + C::NQB;
    uint64_t* v_full = k_full + C::R;
    uint64_t* k_ready = v_full + C::R;
    uint64_t* k_empty = k_ready + C::R;  // K slot free: the last QK reading it has completed
    uint64_t* v_empty = k_empty + C::R;  // V slot free: the last PV reading it has completed
    uint64_t* s_full = v_empty + C::R;
    uint64_t* p_ready = s_full + 2;
    uint64_t* s_empty = p_ready + 2;
    uint64_t* o_full = s_empty + 2;
    uint64_t* o_empty = o_full + 1;
    uint64_t* drain = o_empty + 1;
    uint64_t* drain2 = drain + 1;
    uint64_t* out_ready = drain2 + 1;  // [NQB] the 128 epilogue threads wrote the tile in that buffer
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    float* wq_s = reinterpret_cast<float*>(smem + C::OFF_W);
    float* wk_s = wq_s + D;
    float* rf_s = reinterpret_cast<float*>(smem + C::OFF_R);  // [0, 64) f_hi, [64, 128) f_lo

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long total = static_cast<long long>(p.B) * p.Hkv * p.n_ltiles;
    const long long t_begin = total * blockIdx.x / gridDim.x;
    const long long t_end = total * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        *abort_flag = (smem_u32(smem) & 1023u) == 0 ? 0 : 1;
        if (*abort_flag) report(p.ctl, 30, kErrAlign);
        for (int i = 0; i < C::NQB; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_ready[i], 256);
            mbar_init(&g_full[i], 1);
        }
        for (int i = 0; i < C::R; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_ready[i], 64);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_ready[i], 128);
            mbar_init(&s_empty[i], 1);
        }
        mbar_init(o_full, 1);
        mbar_init(o_empty, 128);
        mbar_init(drain, 1);
        mbar_init(drain2, 1);
        for (int i = 0; i < C::NQB; ++i) mbar_init(&out_ready[i], 128);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    for (int e = threadIdx.x; e < 2 * D; e += kThreads) wq_s[e] = e < D ? __ldg(p.wq + e) : __ldg(p.wk + e - D);
    stage_rope(p.rope, rf_s, rf_s + kMaxRotHalf);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t sbase = smem_u32(smem);
    uint8_t* qbuf0 = smem + C::OFF_Q;
    uint8_t* kring = smem + C::OFF_K;
    uint8_t* vring = smem + C::OFF_V;
    auto aborted = [&]() { return *abort_flag != 0; };
    auto fail = [&]() { *abort_flag = 1; };
    const TileIdx first = decode_tile(t_begin, p.n_ltiles, p.Hkv);
    const int n_tiles = static_cast<int>(t_end - t_begin);

    // QK(n) = Q K^T over the tile's key window into S buffer n&1 (fp16, M128 x N=NK, split
    // in two where the window wraps around the key ring); issued by one thread, which then
    // commits: S ready, and the K slots no later QK of the span reads (the oldest slot, or
    // all of them at the span's end).
    auto issue_qk = [&](int n, int cn, bool span_last) {
        const int sb = n & 1;
        const int row0 = ((cn - C::WS) % C::R) * C::T;
        const int n1 = min(C::NK, C::RR - row0);
        const int n2 = C::NK - n1;
        const uint32_t id1 = idesc_f16_f32(128, n1, false, false);
        const uint32_t id2 = idesc_f16_f32(128, n2 > 0 ? n2 : 16, false, false);
        const uint32_t qofs = C::OFF_Q + (n % C::NQB) * C::QBUF;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t co = (ks >> 2) * C::QCH + (ks & 3) * 32;
            const uint32_t cok = (ks >> 2) * C::KCH + (ks & 3) * 32;
            const uint64_t a = sdesc(sbase + qofs + co, 16, 1024, kSw128);
            umma_bf16(tbase + sb * C::SCOLS, a, sdesc(sbase + C::OFF_K + row0 * 128 + cok, 16, 1024, kSw128), id1,
                      ks > 0);
            if (n2 > 0)
                umma_bf16(tbase + sb * C::SCOLS + n1, a, sdesc(sbase + C::OFF_K + cok, 16, 1024, kSw128), id2, ks > 0);
        }
        umma_commit(&s_full[sb]);
        for (int j = cn - C::WS; j <= (span_last ? cn : cn - C::WS); ++j) umma_commit(&k_empty[j % C::R]);
    };
    // PV(n): O = P V with P read from TMEM (packed bf16, over S buffer n&1) and V from the
    // ring (MN-major).
    auto issue_pv = [&](int n, int cn, bool span_last) {
        const int sb = n & 1;
        const int row0 = ((cn - C::WS) % C::R) * C::T;
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
#pragma unroll
        for (int ks = 0; ks < C::NK / 16; ++ks) {
            const int row = (row0 + ks * 16) % C::RR;
            const uint64_t bd = sdesc(sbase + C::OFF_V + row * 128, C::KCH, 1024, kSw128);
            umma_tmem_a(tbase + C::O_COL, tbase + sb * C::SCOLS + ks * 8, bd, idesc_pv, ks > 0);
        }

        umma_commit(o_full);
        umma_commit(&s_empty[sb]);
        for (int j = cn - C::WS; j <= (span_last ? cn : cn - C::WS); ++j) umma_commit(&v_empty[j % C::R]);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA loop (one thread)
        // Four independent streams, each advanced whenever its next step is possible, so
        // no stream ever waits behind another: K slots (refilled once the last QK reading
        // them has completed), V slots (after the last PV), Q tiles into the 4-deep buffer
        // ring, output stores.  A Q buffer takes the next Q tile once the store of the
        // tile that last held it has been read.
        if (lane == 0 && !aborted()) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            tma_prefetch_desc(&p.tm_out);
            SlotCursor kcur, vcur;
            kcur.init(first, C::WS);
            vcur.init(first, C::WS);
            int nq = 0, ns = 0;
            TileIdx tq = first, ts = first;
            long long t_prog = clock64();
            while (!aborted()) {
                bool prog = false, pending = false;
                for (int kv = 0; kv < 2; ++kv) {
                    SlotCursor& cur = kv == 0 ? kcur : vcur;
                    if (cur.it >= n_tiles) continue;
                    pending = true;
                    const int s = cur.c % C::R;
                    uint64_t* empty = kv == 0 ? &k_empty[s] : &v_empty[s];
                    if (!mbar_test(empty, ((cur.c / C::R) & 1) ^ 1)) continue;
                    uint64_t* full = kv == 0 ? &k_full[s] : &v_full[s];
                    uint8_t* ring = kv == 0 ? kring : vring;
                    const CUtensorMap* map = kv == 0 ? &p.tm_k : &p.tm_v;
                    mbar_arrive_expect_tx(full, C::SLOT_BYTES);
#pragma unroll
                    for (int ch = 0; ch < C::NCH; ++ch)
                        tma_load_4d(ring + ch * C::KCH + s * C::T * 128, map, full, ch * 64, cur.ti.g,
                                    cur.slot_tile() * C::T, cur.ti.b);
                    cur.advance(n_tiles, p.n_ltiles, p.Hkv, C::WS);
                    prog = true;
                }
                if (nq < n_tiles) {
                    pending = true;
                    const int prev_user = nq - C::NQB;  // tile whose output last used this buffer
                    if (prev_user < 0 || ns > prev_user) {
                        if (prev_user >= 0) bulk_wait_read_at_most(ns - 1 - prev_user);
                        const int qb = nq % C::NQB;
                        uint8_t* dst = qbuf0 + qb * C::QBUF;
                        mbar_arrive_expect_tx(&q_full[qb], C::QBUF);
#pragma unroll
                        for (int ch = 0; ch < C::NCH; ++ch)
                            tma_load_4d(dst + ch * C::QCH, &p.tm_q, &q_full[qb], ch * 64, tq.g * G, tq.lt * C::T, tq.b);
                        ++nq;
                        next_tile(tq, p.n_ltiles, p.Hkv);
                        prog = true;
                    }
                }
                if (ns < n_tiles) {
                    pending = true;
                    const int qb = ns % C::NQB;
                    if (mbar_test(&out_ready[qb], (ns / C::NQB) & 1)) {
                        uint8_t* buf = qbuf0 + qb * C::QBUF;
#pragma unroll
                        for (int ch = 0; ch < C::NCH; ++ch)
                            tma_store_4d(&p.tm_out, buf + ch * C::QCH, ch * 64, ts.g * G, ts.lt * C::T, ts.b);
                        bulk_commit();
                        ++ns;
                        next_tile(ts, p.n_ltiles, p.Hkv);
                        prog = true;
                    }
                }
                if (!pending) break;
                const long long now = clock64();
                if (prog) {
                    t_prog = now;
                } else if (now - t_prog > wait_limit_cycles(p.ctl)) {
                    report(p.ctl, 31, kErrTimeout);
                    fail();
                    break;
                }
            }
            bulk_wait_all();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA loop (one thread)
        // QK(n) and PV(m) are issued as soon as their inputs are ready, in tile order each.
        if (lane == 0 && !aborted()) {
            int nqk = 0, npv = 0, cqk = 0, cpv = 0, cqk_cur = 0, cpv_cur = 0;
            TileIdx tqk = first, tpv = first;
            bool qk_have = false, pv_have = false;
            long long t_prog = clock64();
            bool ok = true;
            while (ok && !aborted() && npv < n_tiles) {
                bool prog = false;
                if (nqk < n_tiles) {
                    if (!qk_have) {
                        if (nqk == 0 || tqk.lt == 0) cqk += C::WS;
                        cqk_cur = cqk++;
                        qk_have = true;
                    }
                    const int cn = cqk_cur;
                    const int sb = nqk & 1;
                    bool ready = mbar_test(&s_empty[sb], ((nqk >> 1) & 1) ^ 1) &&
                                 mbar_test(&q_ready[nqk % C::NQB], (nqk / C::NQB) & 1);
                    for (int j = cn - C::WS; j <= cn && ready; ++j) ready = mbar_test(&k_ready[j % C::R], (j / C::R) & 1);
                    if (ready) {
                        tc_fence_after();
                        issue_qk(nqk, cn, nqk + 1 == n_tiles || tqk.lt + 1 == p.n_ltiles);
                        ++nqk;
                        next_tile(tqk, p.n_ltiles, p.Hkv);
                        qk_have = false;
                        prog = true;
                    }
                }
                if (npv < nqk) {
                    if (!pv_have) {
                        if (npv == 0 || tpv.lt == 0) cpv += C::WS;
                        cpv_cur = cpv++;
                        pv_have = true;
                    }
                    const int cn = cpv_cur;
                    const int sb = npv & 1;
                    bool ready = mbar_test(&p_ready[sb], (npv >> 1) & 1) && mbar_test(o_empty, (npv & 1) ^ 1);
                    for (int j = cn - C::WS; j <= cn && ready; ++j) ready = mbar_test(&v_full[j % C::R], (j / C::R) & 1);
                    if (ready) {
                        tc_fence_after();
                        issue_pv(npv, cn, npv + 1 == n_tiles || tpv.lt + 1 == p.n_ltiles);
                        ++npv;
                        next_tile(tpv, p.n_ltiles, p.Hkv);
                        pv_have = false;
                        prog = true;
                    }
                }
                const long long now = clock64();
                if (prog) {
                    t_prog = now;
                } else if (now - t_prog > wait_limit_cycles(p.ctl)) {
                    report(p.ctl, 37, kErrTimeout);
                    ok = false;
                }
            }
            if (!ok) fail();
            // every MMA issued above has completed before the CTA may release TMEM
            umma_commit(drain);
            (void)mbar_wait(drain, 0, p.ctl, 40);
        }
    } else if (warp >= 4 && warp <= 11) {
        // ------------------------------------------------------------ Q transform (2 lanes per row)
        const int row = (threadIdx.x - 128) >> 1;
        int n = 0;
        TileIdx ti = first;
        // position of this row's token, fetched one tile ahead
        auto qpos = [&](const TileIdx& t) {
            const int tok = t.lt * C::T + row / G;
            const long long pi = static_cast<long long>(t.b) * p.L + tok;
            return tok < p.L && idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 84) ? __ldg(p.pos + pi) : 0;
        };
        int pos_next = n_tiles > 0 ? qpos(ti) : 0;
        for (int it = 0; it < n_tiles; ++it, next_tile(ti, p.n_ltiles, p.Hkv)) {
            if (aborted()) break;
            const int pos = pos_next;
            if (it + 1 < n_tiles) {
                TileIdx tn = ti;
                next_tile(tn, p.n_ltiles, p.Hkv);
                pos_next = qpos(tn);
            }
            const int qb = n % C::NQB;
            if (!__all_sync(0xffffffffu, mbar_wait(&q_full[qb], (n / C::NQB) & 1, p.ctl, 41))) {
                fail();
                break;
            }
            if constexpr (PRE)
                (void)pos;
            else if constexpr (ROT > 0)
                qk_norm_rope_row_pair_ct<D, 2 * G, ROT / 2>(qbuf0 + qb * C::QBUF, C::QCH, row, wq_s, p.eps, pos, rf_s,
                                                            rf_s + kMaxRotHalf);
            else
                qk_norm_rope_row_pair<D, 2 * G>(qbuf0 + qb * C::QBUF, C::QCH, row, wq_s, p.eps, pos, p.rope.half, rf_s,
                                                rf_s + kMaxRotHalf);
            fence_async_smem();
            mbar_arrive(&q_ready[qb]);
            ++n;
        }
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------ K transform (2 lanes per row)
        const int kt = threadIdx.x - 64;  // 0..63
        int c = 0;
        bool ok = true;
        auto kslot = [&](int cc, const TileIdx& ti, int tile_l) {
            const int s = cc % C::R;
            // positions first: their latency overlaps the wait for the slot
            int posr[(C::T + 31) / 32];
#pragma unroll
            for (int q = 0; q < (C::T + 31) / 32; ++q) {
                const int r = min(q * 32 + (kt >> 1), C::T - 1);
                const int tok = tile_l * C::T + r;
                const long long pi = static_cast<long long>(ti.b) * p.L + tok;
                posr[q] = (tok >= 0 && tok < p.L && idx_ok(p.ctl, pi, static_cast<long long>(p.B) * p.L, 85))
                              ? __ldg(p.pos + pi)
                              : 0;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&k_full[s], (cc / C::R) & 1, p.ctl, 42))) return false;
#pragma unroll
            for (int r0 = 0; r0 < C::T; r0 += 32) {
                // every lane joins (the row transform is warp-collective); lanes past T only
                // read row T-1 and write nothing
                const bool active = r0 + (kt >> 1) < C::T;
                const int r = min(r0 + (kt >> 1), C::T - 1);
                const int pos = posr[r0 / 32];
                if constexpr (PRE)
                    (void)pos;
                else if constexpr (ROT > 0)
                    qk_norm_rope_row_pair_ct<D, 2, ROT / 2>(kring, C::KCH, s * C::T + r, wk_s, p.eps, pos, rf_s, rf_s + kMaxRotHalf,
                                                            active);
                else
                    qk_norm_rope_row_pair<D, 2>(kring, C::KCH, s * C::T + r, wk_s, p.eps, pos, p.rope.half, rf_s,
                                                    rf_s + kMaxRotHalf, active);
            }
            fence_async_smem();
            mbar_arrive(&k_ready[s]);
            return true;
        };
        TileIdx ti = first;
        for (int it = 0; it < n_tiles && ok; ++it, next_tile(ti, p.n_ltiles, p.Hkv)) {
            if (aborted()) break;
            if (it == 0 || ti.lt == 0)
                for (int w = C::WS; w >= 1 && ok; --w) ok = kslot(c++, ti, ti.lt - w);
            ok = ok && kslot(c++, ti, ti.lt);
        }
        if (!ok) fail();
    } else if (warp >= 12 && warp <= 15) {
        // ------------------------------------------------------------ softmax
        // Scores are bounded: |q_hat| <= sqrt(D) max|wq| and |k_hat| <= sqrt(D) max|wk| after
        // RMSNorm (RoPE keeps norms), so s / sqrt(D) <= sqrt(D) max|wq| max|wk| =: bound.
        // softmax is unchanged by the constant subtracted before exp, so one pass with
        // m = bound needs no row maximum; p = 2^((s - bound) * log2e / sqrt(D)) stays in
        // (2^-2b, 1], far from fp32 / bf16 underflow while 2b < 100 (else the exact
        // two-pass maximum is used).
        const int row = threadIdx.x - 384;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float wqm = 0.f, wkm = 0.f;
        for (int e = lane; e < D; e += 32) {
            wqm = fmaxf(wqm, fabsf(wq_s[e]));
            wkm = fmaxf(wkm, fabsf(wk_s[e]));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            wqm = fmaxf(wqm, __shfl_xor_sync(0xffffffffu, wqm, o));
            wkm = fmaxf(wkm, __shfl_xor_sync(0xffffffffu, wkm, o));
        }
        // fp16 rounding of q_hat / k_hat can exceed the exact bound by ~2^-10 relative
        const float bound = sqrtf(static_cast<float>(D)) * wqm * wkm * 1.002f * p.scale_log2 *
                            sqrtf(static_cast<float>(D));
        const bool use_bound = bound < 50.f;  // log2 units: p >= 2^-100
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        int n = 0;
        TileIdx ti = first;
        for (int it = 0; it < n_tiles; ++it, next_tile(ti, p.n_ltiles, p.Hkv)) {
            if (aborted()) break;
            const int sb = n & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (n >> 1) & 1, p.ctl, 43))) {
                fail();
                break;
            }
            tc_fence_after();
            if (row == 0) {
                // QK(n) has completed: the Q buffer is free for the gate tile the epilogue needs
                const int qb = n % C::NQB;
                uint8_t* dst = qbuf0 + qb * C::QBUF;
                mbar_arrive_expect_tx(&g_full[qb], C::QBUF);
#pragma unroll
                for (int ch = 0; ch < C::NCH; ++ch)
                    tma_load_4d(dst + ch * C::QCH, &p.tm_gate, &g_full[qb], ch * 64, ti.g * G, ti.lt * C::T, ti.b);
            }
            const int i0 = ti.lt * C::T;
            const int tt = row / G;
            // key column kr <-> key i0 - 128 + kr; valid: kr in [max(128 - i0, tt + 129 - W), tt + 128]
            const int kr_lo = max(128 - i0, tt + 129 - p.window);
            const int kr_hi = tt + 128;
            const uint32_t s_addr = lane_addr + sb * C::SCOLS;
            float mb = bound;
            if (!use_bound) {
                float m = -INFINITY;
#pragma unroll 1
                for (int cb = 0; cb < C::NK; cb += 32) {
                    uint32_t r[32];
                    tmem_ld32(s_addr + cb, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (cb + k >= kr_lo && cb + k <= kr_hi) m = fmaxf(m, __uint_as_float(r[k]));
                }
                mb = (m == -INFINITY ? 0.f : m) * p.scale_log2;
            }
            const float2 nm2 = make_float2(-mb, -mb);
            float2 lacc = make_float2(0.f, 0.f), lacc2 = make_float2(0.f, 0.f);
            // one code path for every 16-column group, with the window test per element: the kernel's
            // six warp roles run concurrently, and a second (unmasked) copy of this body cost more in
            // instruction fetch than the tests it saves
            auto soft16 = [&](const uint32_t* r, int cb) {
                uint32_t pk[8];
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    const float2 x = fma2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), sc2, nm2);
                    const int kr = cb + k;
                    const float e0 = (kr >= kr_lo && kr <= kr_hi) ? ex2_approx(x.x) : 0.f;
                    const float e1 = (kr + 1 >= kr_lo && kr + 1 <= kr_hi) ? ex2_approx(x.y) : 0.f;
                    pk[k / 2] = pack_bf16x2(e0, e1);
                }
                // row sums of the very bf16 P the PV product uses
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    acc_bf16x2(pk[k], lacc.x, lacc.y);
                    acc_bf16x2(pk[k + 1], lacc2.x, lacc2.y);
                }
                // P (keys cb..cb+15) -> TMEM columns cb/2 .. cb/2+7 of this S buffer (already read)
                tmem_st8(s_addr + cb / 2, pk);
            };
#pragma unroll 1
            for (int cb = 0; cb < C::NK; cb += 16) {
                uint32_t ra[16];
                tmem_ld16(s_addr + cb, ra);
                tmem_wait_ld();
                soft16(ra, cb);
            }
            {
                uint32_t lv[8];
                const float lsum = (lacc.x + lacc.y) + (lacc2.x + lacc2.y);
#pragma unroll
                for (int k = 0; k < 8; ++k) lv[k] = __float_as_uint(lsum);
                // l for the epilogue, four tiles deep: slot n & 3 is rewritten only by the
                // softmax of tile n + 4, whose S needs PV(n + 2), which waits for the
                // epilogue of tile n + 1 and so for that of tile n
                tmem_st8(lane_addr + C::L_COL + (n & 3) * 8, lv);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_ready[sb]);
            ++n;
        }
    } else if (warp >= 16 && warp <= 19) {
        // ------------------------------------------------------------ epilogue
        const int row = threadIdx.x - 512;
        const uint32_t lane_addr = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        int n = 0;
        TileIdx ti = first;
        for (int it = 0; it < n_tiles; ++it, next_tile(ti, p.n_ltiles, p.Hkv)) {
            if (aborted()) break;
            const int qb = n % C::NQB;
            bool ok = mbar_wait(o_full, n & 1, p.ctl, 45) && mbar_wait(&g_full[qb], (n / C::NQB) & 1, p.ctl, 47);
            if (!__all_sync(0xffffffffu, ok)) {
                fail();
                break;
            }
            tc_fence_after();
            uint32_t lraw;
            tmem_ld1(lane_addr + C::L_COL + (n & 3) * 8, lraw);
            uint32_t ra[16], rb[16];
            tmem_ld16(lane_addr + C::O_COL, ra);
            tmem_wait_ld();
            const float lsum = __uint_as_float(lraw);
            // out = O / l * sigmoid(g) in fp32, as O / (l (1 + 2^(-g log2 e))): one reciprocal per
            // element for 1/l and the sigmoid together, with no cancellation for g < 0; a row with
            // l = 0 has O = 0, and l = 1 there keeps the product finite.  PRE: sigmoid(g) is given.
            const float c = lsum > 0.f ? 1.0f / lsum : 0.f;
            const float2 c2 = make_float2(c, c);
            const float ls = lsum > 0.f ? lsum : 1.f;
            const float2 l2 = make_float2(ls, ls);
            uint8_t* buf = qbuf0 + qb * C::QBUF;
            auto epi16 = [&](const uint32_t* r, int cb) {
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    const int e0 = cb + q2 * 8;
                    uint8_t* gp = buf + (e0 >> 6) * C::QCH + sw128_off(row, (e0 & 63) >> 3);
                    const uint4 gv = *reinterpret_cast<const uint4*>(gp);
                    const uint32_t gu[4] = {gv.x, gv.y, gv.z, gv.w};
                    uint32_t ou[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 rr = make_float2(__uint_as_float(r[q2 * 8 + 2 * k]), __uint_as_float(r[q2 * 8 + 2 * k + 1]));
                        float2 o;
                        if constexpr (PRE) {
                            o = mul2(mul2(rr, c2), bf2f2(gu[k]));
                        } else {
                            const float2 t = mul2(bf2f2(gu[k]), make_float2(-kLog2e, -kLog2e));
                            const float2 d = fma2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), l2, l2);
                            o = mul2(rr, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
                        }
                        ou[k] = pack_bf16x2(o.x, o.y);
                    }
                    *reinterpret_cast<uint4*>(gp) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                }
            };
#pragma unroll 1
            for (int cb = 0; cb < D; cb += 32) {
                tmem_ld16(lane_addr + C::O_COL + cb + 16, rb);
                epi16(ra, cb);
                tmem_wait_ld();
                if (cb + 32 < D) tmem_ld16(lane_addr + C::O_COL + cb + 32, ra);
                epi16(rb, cb + 16);
                tmem_wait_ld();
            }
            tc_fence_before();
            mbar_arrive(o_empty);
            fence_async_smem();  // output visible to the TMA store issued by the TMA loop
            mbar_arrive(&out_ready[qb]);
            ++n;
        }
    }
    __syncthreads();
    if (aborted() && threadIdx.x == 0) {
        // abandoned run: give copies still in flight time to land before shared memory is released
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
    }
    tc_fence_after();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, C::TMEM_COLS);
}

template <int D, int G, int ROT, bool PRE = false>
cudaError_t launch_t(const PrefillParams& p, cudaStream_t s) {
    using C = Swa2<D, G>;
    auto k = swa2_kernel<D, G, ROT, PRE>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long tiles = static_cast<long long>(p.B) * p.Hkv * p.n_ltiles;
    const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
    k<<<grid, kThreads, C::SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

// GQA 4 and 8; GQA 1 and 2 (whose score tiles leave no TMEM for double buffering)
// take the one-tile kernel in swa_prefill.cu.
bool swa2_supports(int d, int G) { return (d == 64 || d == 128) && (G == 4 || G == 8); }

// The rotary widths of rotary ratio 0.33 (2 * floor(0.33 * d / 2)) get kernels with the
// width compiled in; any other width takes the general kernel.
template <int D, int G>
cudaError_t launch_rot(const PrefillParams& p, cudaStream_t s) {
    constexpr int ROT_STD = D == 128 ? 42 : 20;
    if (p.pre) return launch_t<D, G, 0, true>(p, s);
    if (2 * p.rope.half == ROT_STD) return launch_t<D, G, ROT_STD>(p, s);
    return launch_t<D, G, 0>(p, s);
}

cudaError_t launch_swa2_prefill(const PrefillParams& p, int d, cudaStream_t s) {
    const int G = p.Hq / p.Hkv;
    if (d == 128 && G == 4) return launch_rot<128, 4>(p, s);
    if (d == 64 && G == 4) return launch_rot<64, 4>(p, s);
    if (d == 128 && G == 8) return launch_rot<128, 8>(p, s);
    if (d == 64 && G == 8) return launch_rot<64, 8>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace zg
