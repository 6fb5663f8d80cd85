// api.cu -- the C ABI declared in include/zg_attn.h: argument checks, TMA
// descriptors, RoPE constants, launches.  No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/zg_attn.h"
#include "zg_kernels.cuh"

namespace zg {

// device error word (bounded waits record themselves here)
__device__ uint32_t g_err_word = 0;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

unsigned long long wait_limit_ns() {
    static unsigned long long lim = [] {
        const char* e = std::getenv("ZG_WAIT_LIMIT_NS");
        unsigned long long v = e ? std::strtoull(e, nullptr, 10) : 0ull;
        return v ? v : 4000000000ull;
    }();
    return lim;
}

bool dev_ctl(DevCtl& ctl) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return false;
    ctl.err_word = static_cast<uint32_t*>(p);
    ctl.wait_limit_ns = wait_limit_ns();
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D bf16 tensor map over [outer][L][heads][d] with a {64, box_heads, box_rows, 1} box, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int d, int heads, int L, int B, int box_heads, int box_rows,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2, (cuuint64_t)L * heads * d * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D tensor map of one-byte elements (E4M3) over a row-major [d3][d2][d1][d0] array, 128-byte swizzle
bool make_map_u8(CUtensorMap* m, const void* base, long long d0, long long d1, long long d2, long long d3,
                 uint32_t b0, uint32_t b1, uint32_t b2) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2, (cuuint64_t)d3};
    cuuint64_t strides[3] = {(cuuint64_t)d0, (cuuint64_t)(d0 * d1), (cuuint64_t)(d0 * d1 * d2)};
    cuuint32_t box[4] = {b0, b1, b2, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D fp32 tensor map over [outer][L][heads][d] with a {32, box_heads, box_rows, 1} box (128 bytes
// inner), 128-byte swizzle
bool make_map_f32(CUtensorMap* m, const void* base, int d, int heads, int L, int B, int box_heads, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 4, (cuuint64_t)heads * d * 4, (cuuint64_t)L * heads * d * 4};
    cuuint32_t box[4] = {32, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map over a decode cache [slices][rows][d] (bf16, or E4M3 bytes when fp8) with a
// {min(d * elem, 128 B), box_rows, 1} box and the 128-byte (64-byte for 64-byte rows) swizzle
bool make_cache_map(CUtensorMap* m, const void* base, int d, long long rows, long long slices, bool fp8,
                    int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const int eb = fp8 ? 1 : 2;
    const int row_bytes = d * eb;
    const int box_bytes = row_bytes < 128 ? row_bytes : 128;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)slices};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows * row_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(box_bytes / eb), (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// theta^(-2j/r) in double, split into float head + float tail
bool rope_consts(RopeConsts& rc, int rotary_dim, double theta) {
    if (rotary_dim < 0 || (rotary_dim & 1) || rotary_dim / 2 > kMaxRotHalf) return false;
    rc.half = rotary_dim / 2;
    for (int j = 0; j < kMaxRotHalf; ++j) {
        double f = j < rc.half ? std::pow(theta, -2.0 * j / rotary_dim) : 0.0;
        float hi = static_cast<float>(f);
        rc.f_hi[j] = hi;
        rc.f_lo[j] = static_cast<float>(f - static_cast<double>(hi));
    }
    return true;
}

zg_status check_prefill(const void* q, const void* k, const void* v, const void* gate, bool gated, const void* pos,
                        const void* wq, const void* wk, const void* out, int B, int L, int Hq, int Hkv, int d,
                        int rotary_dim, double theta, float eps) {
    if (!q || !k || !v || (gated && !gate) || !pos || !wq || !wk || !out) return ZG_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (gated && !aligned16(gate)) || !aligned16(pos) ||
        !aligned16(wq) || !aligned16(wk) || !aligned16(out))
        return ZG_ERR_ALIGN;
    if (B < 0 || L < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return ZG_ERR_SHAPE;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1)) return ZG_ERR_SHAPE;
    if (!(theta > 0.0) || !(eps >= 0.0f)) return ZG_ERR_SHAPE;
    return ZG_OK;
}

}  // namespace
}  // namespace zg

namespace zg {
namespace {
// ---------------------------------------------------------------- prefill + decode caches
// host checks of the cache arguments (done before anything is launched)
zg_status check_cache(const void* ck, const void* cv, int d, long long S) {
    if (!ck || !cv) return ZG_ERR_NULL;
    if (!aligned16(ck) || !aligned16(cv)) return ZG_ERR_ALIGN;
    if (S < 1) return ZG_ERR_SHAPE;
    if (d != 64 && d != 128) return ZG_ERR_UNSUPPORTED;  // the head sizes the decode step reads
    return ZG_OK;
}
zg_status write_cache(const zg_bf16* k, const zg_bf16* v, const int32_t* pos, const float* wk, void* ck,
                      void* cv, int B, int L, int Hkv, int d, long long S, bool ring, int rotary_dim, double theta,
                      float eps, zg_stream stream, int fp8 = 0, float k_scale = 1.0f, float v_scale = 1.0f) {
    if (B == 0 || L == 0) return ZG_OK;
    if (B > 65535 || static_cast<long long>(L) * Hkv >= (1ll << 31) || (ring && S >= (1ll << 31)))
        return ZG_ERR_UNSUPPORTED;
    CacheParams c;
    std::memset(&c, 0, sizeof(c));
    if (!dev_ctl(c.ctl)) return ZG_ERR_CUDA;
    c.k = reinterpret_cast<const __nv_bfloat16*>(k);
    c.v = reinterpret_cast<const __nv_bfloat16*>(v);
    c.pos = pos;
    c.wk = wk;
    c.cache_k = static_cast<__nv_bfloat16*>(ck);  // E4M3 bytes when fp8
    c.cache_v = static_cast<__nv_bfloat16*>(cv);
    c.fp8 = fp8;
    c.k_scale = k_scale;
    c.v_scale = v_scale;
    c.B = B;
    c.L = L;
    c.Hkv = Hkv;
    c.S = S;
    c.ring = ring ? 1 : 0;
    c.i0 = ring && L > S ? static_cast<int>(L - S) : 0;
    c.eps = eps;
    if (!rope_consts(c.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_kv_cache(c, d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}
}  // namespace
}  // namespace zg

namespace zg {
// Every argument check of one decode step except the workspace's, in the order the entry points
// report them; *ng receives the number of global layers.  Shared by zg_hybrid_decode(_fp8) and
// the allocation-free entry point, so a bad call gets the same status from each.
int hybrid_decode_check(const void* q, const void* k_new, const void* v_new, const void* gate, const void* pos,
                        const void* wq, const void* wk, const uint8_t* is_global, const void* k_glob,
                        const void* v_glob, const void* k_ring, const void* v_ring, const void* out, int NL, int B,
                        int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim, double theta, float eps,
                        int fp8, float k_scale, float v_scale, int* ng) {
    if (!q || !k_new || !v_new || !gate || !pos || !wq || !wk || !is_global || !out) return ZG_ERR_NULL;
    if (fp8 && !(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
        return ZG_ERR_SHAPE;
    if (NL < 0 || B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv || window <= 0) return ZG_ERR_SHAPE;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1) || !(theta > 0.0) || !(eps >= 0.0f)) return ZG_ERR_SHAPE;
    if (NL > kMaxLayers) return ZG_ERR_UNSUPPORTED;
    int NG = 0;
    for (int l = 0; l < NL; ++l) NG += is_global[l] ? 1 : 0;
    const int NS = NL - NG;
    if ((NG && (!k_glob || !v_glob)) || (NS && (!k_ring || !v_ring))) return ZG_ERR_NULL;
    const void* ptrs[] = {q, k_new, v_new, gate, pos, wq, wk, out};
    for (const void* x : ptrs)
        if (!aligned16(x)) return ZG_ERR_ALIGN;
    if ((NG && (!aligned16(k_glob) || !aligned16(v_glob))) || (NS && (!aligned16(k_ring) || !aligned16(v_ring))))
        return ZG_ERR_ALIGN;
    if (NG && S_max <= 0) return ZG_ERR_SHAPE;
    if (!decode_supports(d, Hq / Hkv) || window > 4096 || S_max >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    const long long nsplit = NG ? (S_max + kDecodeSplitLen - 1) / kDecodeSplitLen : 1;
    const long long ctas = static_cast<long long>(NG) * B * Hkv * nsplit + static_cast<long long>(NS) * B * Hkv;
    if (ctas >= (1ll << 31) || static_cast<long long>(NG) * B * Hq >= (1ll << 31) ||
        static_cast<long long>(NL) * B * Hkv >= (1ll << 31))
        return ZG_ERR_UNSUPPORTED;
    *ng = NG;
    return ZG_OK;
}
}  // namespace zg

using namespace zg;

extern "C" {

zg_status zg_swa_prefill(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const zg_bf16* gate,
                         const int32_t* pos, const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq,
                         int Hkv, int d, int window, int rotary_dim, double theta, float eps, zg_stream stream) {
    zg_status st = check_prefill(q, k, v, gate, true, pos, wq, wk, out, B, L, Hq, Hkv, d, rotary_dim, theta, eps);
    if (st != ZG_OK) return st;
    if (window < 1) return ZG_ERR_SHAPE;
    const int G = Hq / Hkv;
    if ((d != 64 && d != 128) || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) || window > 128 || Hkv > 65535)
        return ZG_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return ZG_OK;
    const int T = 128 / G;
    const long long n_lt = (L + T - 1) / T;
    if (n_lt * Hkv * B >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    const int NK = swa_kv_box_rows(G);

    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    if (!dev_ctl(p.ctl)) return ZG_ERR_CUDA;
    if (!make_map(&p.tm_q, q, d, Hq, L, B, G, T) || !make_map(&p.tm_gate, gate, d, Hq, L, B, G, T) ||
        !make_map(&p.tm_out, out, d, Hq, L, B, G, T) || !make_map(&p.tm_k, k, d, Hkv, L, B, 1, NK) ||
        !make_map(&p.tm_v, v, d, Hkv, L, B, 1, NK))
        return ZG_ERR_CUDA;
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = window;
    p.n_ltiles = static_cast<int>(n_lt);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    if (!rope_consts(p.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_swa_prefill(p, d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

size_t zg_global_prefill_workspace_bytes(int B, int L, int Hkv, int d) {
    if (B <= 0 || L <= 0 || Hkv <= 0 || d <= 0) return 0;
    return static_cast<size_t>(B) * L * Hkv * d * 2;  // fp16 normalised + rotated keys
}

zg_status zg_global_prefill(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const int32_t* pos,
                            const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq, int Hkv, int d,
                            int rotary_dim, double theta, float eps, void* workspace, size_t workspace_bytes,
                            zg_stream stream) {
    zg_status st = check_prefill(q, k, v, nullptr, false, pos, wq, wk, out, B, L, Hq, Hkv, d, rotary_dim, theta, eps);
    if (st != ZG_OK) return st;
    const int G = Hq / Hkv;
    if (!global_supports(d, G) || Hkv > 65535) return ZG_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return ZG_OK;
    const size_t need = zg_global_prefill_workspace_bytes(B, L, Hkv, d);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ZG_ERR_WORKSPACE;
    const int T = global_q_tile_tokens(G);
    const long long n_lt = (L + T - 1) / T;
    if (n_lt * Hkv * B >= (1ll << 31) || static_cast<long long>(B) * L * Hkv / 8 >= (1ll << 31))
        return ZG_ERR_UNSUPPORTED;

    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    if (!dev_ctl(p.ctl)) return ZG_ERR_CUDA;
    if (!make_map(&p.tm_q, q, d, Hq, L, B, G, T) || !make_map(&p.tm_out, out, d, Hq, L, B, G, T) ||
        !make_map(&p.tm_kh, workspace, d, Hkv, L, B, 1, 128, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
        !make_map(&p.tm_v, v, d, Hkv, L, B, 1, 128))
        return ZG_ERR_CUDA;
    p.k_raw = k;
    p.khat = workspace;
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = L;
    p.n_ltiles = static_cast<int>(n_lt);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    if (!rope_consts(p.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_global_prefill(p, d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

size_t zg_global_prefill_fp8_workspace_bytes(int B, int L, int Hkv, int d) {
    if (B <= 0 || L <= 0 || Hkv <= 0 || d <= 0) return 0;
    const size_t lp = (static_cast<size_t>(L) + 15) / 16 * 16;
    return static_cast<size_t>(B) * Hkv * d * (static_cast<size_t>(L) + lp);  // k_hat, then V^T
}

// E4M3 prefill on the global pipeline: the global layer (gate NULL, every earlier key) or the gated
// sliding-window layer (gate given, window >= 1)
static zg_status prefill_fp8(const uint8_t* q, const uint8_t* k, const uint8_t* v, const zg_bf16* gate,
                             const int32_t* pos, const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq,
                             int Hkv, int d, int window, int rotary_dim, double theta, float eps, float q_scale,
                             float k_scale, float v_scale, void* workspace, size_t workspace_bytes, zg_stream stream) {
    const bool swa = gate != nullptr;
    zg_status st = check_prefill(q, k, v, gate, swa, pos, wq, wk, out, B, L, Hq, Hkv, d, rotary_dim, theta, eps);
    if (st != ZG_OK) return st;
    if (swa && window < 1) return ZG_ERR_SHAPE;
    if (!(std::isfinite(q_scale) && q_scale > 0.f && std::isfinite(k_scale) && k_scale > 0.f &&
          std::isfinite(v_scale) && v_scale > 0.f))
        return ZG_ERR_SHAPE;
    const int G = Hq / Hkv;
    if (d != 128 || !global_supports(d, G) || Hkv > 65535) return ZG_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return ZG_OK;
    const size_t need = zg_global_prefill_fp8_workspace_bytes(B, L, Hkv, d);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ZG_ERR_WORKSPACE;
    const int T = global_q_tile_tokens(G);
    const long long n_lt = (L + T - 1) / T;
    if (n_lt * Hkv * B >= (1ll << 31) || static_cast<long long>(B) * L * Hkv / 8 >= (1ll << 31))
        return ZG_ERR_UNSUPPORTED;
    const int lp = (L + 15) / 16 * 16;
    uint8_t* kh = static_cast<uint8_t*>(workspace);
    uint8_t* vt = kh + static_cast<size_t>(B) * L * Hkv * d;
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    if (!dev_ctl(p.ctl)) return ZG_ERR_CUDA;
    if (!make_map_u8(&p.tm_q, q, d, Hq, L, B, 128, G, T) || !make_map(&p.tm_out, out, d, Hq, L, B, G, T) ||
        !make_map_u8(&p.tm_kh, kh, d, Hkv, L, B, 128, 1, 128) || !make_map_u8(&p.tm_vt, vt, lp, d, Hkv, B, 128, 128, 1) ||
        (swa && !make_map(&p.tm_gate, gate, d, Hq, L, B, G, T)))
        return ZG_ERR_CUDA;
    p.fp8 = 1;
    p.swa = swa ? 1 : 0;
    p.k_raw = k;
    p.v_raw = v;
    p.khat = kh;
    p.vt_ws = vt;
    p.vt_lp = lp;
    p.in_dequant_q = 1.0f / q_scale;
    p.in_dequant_k = 1.0f / k_scale;
    p.in_dequant_v = 1.0f / v_scale;
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = swa ? window : L;
    p.n_ltiles = static_cast<int>(n_lt);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    if (!rope_consts(p.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_global_prefill(p, d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

zg_status zg_global_prefill_fp8(const uint8_t* q, const uint8_t* k, const uint8_t* v, const int32_t* pos,
                                const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq, int Hkv,
                                int d, int rotary_dim, double theta, float eps, float q_scale, float k_scale,
                                float v_scale, void* workspace, size_t workspace_bytes, zg_stream stream) {
    return prefill_fp8(q, k, v, nullptr, pos, wq, wk, out, B, L, Hq, Hkv, d, 0, rotary_dim, theta, eps, q_scale, k_scale,
                       v_scale, workspace, workspace_bytes, stream);
}

zg_status zg_swa_prefill_fp8(const uint8_t* q, const uint8_t* k, const uint8_t* v, const zg_bf16* gate,
                             const int32_t* pos, const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq,
                             int Hkv, int d, int window, int rotary_dim, double theta, float eps, float q_scale,
                             float k_scale, float v_scale, void* workspace, size_t workspace_bytes, zg_stream stream) {
    if (!gate) return ZG_ERR_NULL;
    return prefill_fp8(q, k, v, gate, pos, wq, wk, out, B, L, Hq, Hkv, d, window, rotary_dim, theta, eps, q_scale,
                       k_scale, v_scale, workspace, workspace_bytes, stream);
}

zg_status zg_kv_cache_write(const zg_bf16* k, const zg_bf16* v, const int32_t* pos, const float* wk,
                            zg_bf16* k_cache, zg_bf16* v_cache, int B, int L, int Hkv, int d, int64_t S, int ring,
                            int rotary_dim, double theta, float eps, zg_stream stream) {
    if (!k || !v || !pos || !wk) return ZG_ERR_NULL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(pos) || !aligned16(wk)) return ZG_ERR_ALIGN;
    zg_status st = check_cache(k_cache, v_cache, d, S);
    if (st != ZG_OK) return st;
    if (B < 0 || L < 0 || Hkv <= 0 || (ring != 0 && ring != 1)) return ZG_ERR_SHAPE;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1) || !(theta > 0.0) || !(eps >= 0.0f)) return ZG_ERR_SHAPE;
    if (static_cast<long long>(B) * L * Hkv / 8 >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    return write_cache(k, v, pos, wk, k_cache, v_cache, B, L, Hkv, d, S, ring != 0, rotary_dim, theta, eps, stream);
}

zg_status zg_kv_cache_write_fp8(const zg_bf16* k, const zg_bf16* v, const int32_t* pos, const float* wk,
                                uint8_t* k_cache, uint8_t* v_cache, int B, int L, int Hkv, int d, int64_t S, int ring,
                                int rotary_dim, double theta, float eps, float k_scale, float v_scale,
                                zg_stream stream) {
    if (!k || !v || !pos || !wk) return ZG_ERR_NULL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(pos) || !aligned16(wk)) return ZG_ERR_ALIGN;
    zg_status st = check_cache(k_cache, v_cache, d, S);
    if (st != ZG_OK) return st;
    if (B < 0 || L < 0 || Hkv <= 0 || (ring != 0 && ring != 1)) return ZG_ERR_SHAPE;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1) || !(theta > 0.0) || !(eps >= 0.0f)) return ZG_ERR_SHAPE;
    if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f)) return ZG_ERR_SHAPE;
    if (static_cast<long long>(B) * L * Hkv / 8 >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    return write_cache(k, v, pos, wk, k_cache, v_cache, B, L, Hkv, d, S, ring != 0, rotary_dim, theta, eps, stream, 1,
                       k_scale, v_scale);
}

// ---- the gated SWA prefill from host buffers: chunks of tokens pipelined over three streams
namespace {
constexpr int kHostSlots = 2;  // device staging slots (chunk c uses slot c mod 2)
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
struct HostSlotLayout {
    size_t q, k, v, gate, pos, out, bytes;  // offsets inside one slot, and its size
};
HostSlotLayout host_slot_layout(int B, int rows, int Hq, int Hkv, int d) {
    HostSlotLayout s;
    const size_t nq = static_cast<size_t>(B) * rows * Hq * d * 2, nk = static_cast<size_t>(B) * rows * Hkv * d * 2;
    s.q = 0;
    s.gate = s.q + align256(nq);
    s.out = s.gate + align256(nq);
    s.k = s.out + align256(nq);
    s.v = s.k + align256(nk);
    s.pos = s.v + align256(nk);
    s.bytes = s.pos + align256(static_cast<size_t>(B) * rows * 4);
    return s;
}
// halo of earlier keys a chunk carries: the window's W - 1 keys, rounded up to whole 128-token
// blocks so the chunk's query tiles fall where they fall in one unchunked call
int host_halo(int window) { return (window - 1 + 127) / 128 * 128; }
}  // namespace

size_t zg_swa_prefill_host_workspace_bytes(int B, int Hq, int Hkv, int d, int window, int chunk_tokens) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || window < 1 || chunk_tokens <= 0) return 0;
    const int rows = chunk_tokens + host_halo(window);
    return 256 + kHostSlots * host_slot_layout(B, rows, Hq, Hkv, d).bytes + 2 * static_cast<size_t>(d) * 4;
}

zg_status zg_swa_prefill_host(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const zg_bf16* gate,
                              const int32_t* pos, const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq,
                              int Hkv, int d, int window, int rotary_dim, double theta, float eps, int chunk_tokens,
                              void* workspace, size_t workspace_bytes, zg_stream stream) {
    if (!q || !k || !v || !gate || !pos || !wq || !wk || !out) return ZG_ERR_NULL;
    if (B < 0 || L < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv || window < 1 || chunk_tokens <= 0)
        return ZG_ERR_SHAPE;
    if (B == 0 || L == 0) return ZG_OK;
    const size_t need = zg_swa_prefill_host_workspace_bytes(B, Hq, Hkv, d, window, chunk_tokens);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ZG_ERR_WORKSPACE;
    const int halo = host_halo(window);
    const int cap = chunk_tokens + halo;  // rows of one slot
    const HostSlotLayout lay = host_slot_layout(B, cap, Hq, Hkv, d);
    uint8_t* base = static_cast<uint8_t*>(workspace);
    float* wq_d = reinterpret_cast<float*>(base + kHostSlots * lay.bytes);
    float* wk_d = wq_d + d;
    const size_t rq = static_cast<size_t>(Hq) * d * 2, rk = static_cast<size_t>(Hkv) * d * 2;  // bytes per token
    cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
    cudaEvent_t ev[3 * kHostSlots + 2] = {};
    zg_status st = ZG_OK;
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && st == ZG_OK) st = ZG_ERR_CUDA;
        return st == ZG_OK;
    };
    bool good = ok(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking)) &&
                ok(cudaStreamCreateWithFlags(&s_run, cudaStreamNonBlocking)) &&
                ok(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking));
    for (int i = 0; good && i < 3 * kHostSlots + 2; ++i) good = ok(cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
    cudaEvent_t* ev_in = ev;                   // slot inputs copied
    cudaEvent_t* ev_run = ev + kHostSlots;     // slot kernel done
    cudaEvent_t* ev_out = ev + 2 * kHostSlots; // slot output copied back
    cudaEvent_t ev_start = ev[3 * kHostSlots], ev_end = ev[3 * kHostSlots + 1];
    if (good) {  // the internal streams start after the caller's earlier work
        good = ok(cudaEventRecord(ev_start, user)) && ok(cudaStreamWaitEvent(s_in, ev_start, 0)) &&
               ok(cudaStreamWaitEvent(s_run, ev_start, 0)) &&
               ok(cudaMemcpyAsync(wq_d, wq, static_cast<size_t>(d) * 4, cudaMemcpyHostToDevice, s_in)) &&
               ok(cudaMemcpyAsync(wk_d, wk, static_cast<size_t>(d) * 4, cudaMemcpyHostToDevice, s_in));
    }
    const int n_chunks = (L + chunk_tokens - 1) / chunk_tokens;
    for (int c = 0; good && c < n_chunks; ++c) {
        const int sl = c % kHostSlots;
        uint8_t* sb = base + sl * lay.bytes;
        const int t0 = c * chunk_tokens, t1 = std::min(L, t0 + chunk_tokens);
        const int h = std::min(t0, halo), lc = (t1 - t0) + h;
        auto* qd = reinterpret_cast<zg_bf16*>(sb + lay.q);
        auto* gd = reinterpret_cast<zg_bf16*>(sb + lay.gate);
        auto* od = reinterpret_cast<zg_bf16*>(sb + lay.out);
        auto* kd = reinterpret_cast<zg_bf16*>(sb + lay.k);
        auto* vd = reinterpret_cast<zg_bf16*>(sb + lay.v);
        auto* pd = reinterpret_cast<int32_t*>(sb + lay.pos);
        // inputs: keys, values and positions of the halo and the chunk; queries and gate of the chunk
        // (the halo rows' outputs are computed and dropped); the slot's previous kernel must be done
        if (c >= kHostSlots) good = ok(cudaStreamWaitEvent(s_in, ev_run[sl], 0));
        const auto* kh = reinterpret_cast<const uint8_t*>(k);
        const auto* vh = reinterpret_cast<const uint8_t*>(v);
        const auto* qh = reinterpret_cast<const uint8_t*>(q);
        const auto* gh = reinterpret_cast<const uint8_t*>(gate);
        const auto* ph = reinterpret_cast<const uint8_t*>(pos);
        good = good &&
               ok(cudaMemcpy2DAsync(kd, lc * rk, kh + (t0 - h) * rk, L * rk, lc * rk, B, cudaMemcpyHostToDevice, s_in)) &&
               ok(cudaMemcpy2DAsync(vd, lc * rk, vh + (t0 - h) * rk, L * rk, lc * rk, B, cudaMemcpyHostToDevice, s_in)) &&
               ok(cudaMemcpy2DAsync(pd, static_cast<size_t>(lc) * 4, ph + static_cast<size_t>(t0 - h) * 4,
                                    static_cast<size_t>(L) * 4, static_cast<size_t>(lc) * 4, B, cudaMemcpyHostToDevice,
                                    s_in)) &&
               ok(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(qd) + h * rq, lc * rq, qh + t0 * rq, L * rq,
                                    (t1 - t0) * rq, B, cudaMemcpyHostToDevice, s_in)) &&
               ok(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(gd) + h * rq, lc * rq, gh + t0 * rq, L * rq,
                                    (t1 - t0) * rq, B, cudaMemcpyHostToDevice, s_in)) &&
               ok(cudaEventRecord(ev_in[sl], s_in));
        // the kernel, once the inputs are in and the slot's previous output has been copied out
        good = good && ok(cudaStreamWaitEvent(s_run, ev_in[sl], 0)) &&
               (c < kHostSlots || ok(cudaStreamWaitEvent(s_run, ev_out[sl], 0)));
        if (good) {
            const zg_status ks = zg_swa_prefill(qd, kd, vd, gd, pd, wq_d, wk_d, od, B, lc, Hq, Hkv, d, window,
                                                rotary_dim, theta, eps, reinterpret_cast<zg_stream>(s_run));
            if (ks != ZG_OK) {
                st = ks;
                good = false;
            }
        }
        good = good && ok(cudaEventRecord(ev_run[sl], s_run)) && ok(cudaStreamWaitEvent(s_out, ev_run[sl], 0)) &&
               ok(cudaMemcpy2DAsync(reinterpret_cast<uint8_t*>(out) + t0 * rq, L * rq,
                                    reinterpret_cast<uint8_t*>(od) + h * rq, lc * rq, (t1 - t0) * rq, B,
                                    cudaMemcpyDeviceToHost, s_out)) &&
               ok(cudaEventRecord(ev_out[sl], s_out));
    }
    // the caller's stream continues after the last copy back (or after whatever was issued)
    if (s_out && ev_end && cudaEventRecord(ev_end, s_out) == cudaSuccess) (void)cudaStreamWaitEvent(user, ev_end, 0);
    for (auto& e : ev)
        if (e) cudaEventDestroy(e);  // released once their work is done
    for (cudaStream_t x : {s_in, s_run, s_out})
        if (x) cudaStreamDestroy(x);
    return st;
}

zg_status zg_swa_prefill_with_cache(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const zg_bf16* gate,
                                    const int32_t* pos, const float* wq, const float* wk, zg_bf16* out, int B, int L,
                                    int Hq, int Hkv, int d, int window, int rotary_dim, double theta, float eps,
                                    zg_bf16* k_ring, zg_bf16* v_ring, int ring_slots, zg_stream stream) {
    zg_status st = check_cache(k_ring, v_ring, d, ring_slots);
    if (st != ZG_OK) return st;
    st = zg_swa_prefill(q, k, v, gate, pos, wq, wk, out, B, L, Hq, Hkv, d, window, rotary_dim, theta, eps, stream);
    if (st != ZG_OK) return st;
    return write_cache(k, v, pos, wk, k_ring, v_ring, B, L, Hkv, d, ring_slots, true, rotary_dim, theta, eps, stream);
}

zg_status zg_global_prefill_with_cache(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const int32_t* pos,
                                       const float* wq, const float* wk, zg_bf16* out, int B, int L, int Hq, int Hkv,
                                       int d, int rotary_dim, double theta, float eps, void* workspace,
                                       size_t workspace_bytes, zg_bf16* k_cache, zg_bf16* v_cache, int64_t S_max,
                                       zg_stream stream) {
    zg_status st = check_cache(k_cache, v_cache, d, S_max);
    if (st != ZG_OK) return st;
    st = zg_global_prefill(q, k, v, pos, wq, wk, out, B, L, Hq, Hkv, d, rotary_dim, theta, eps, workspace,
                           workspace_bytes, stream);
    if (st != ZG_OK) return st;
    return write_cache(k, v, pos, wk, k_cache, v_cache, B, L, Hkv, d, S_max, false, rotary_dim, theta, eps, stream);
}

// ---------------------------------------------------------------- projections and the whole gated SWA layer
namespace {
// 2-D bf16 tensor map over a row-major [outer][inner] matrix, {64, box_outer} box, 128-byte swizzle
bool make_map_2d(CUtensorMap* m, const void* base, long long inner, long long outer, int box_outer) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Proj {
    const void* w;  // W [K, n]
    void* y;        // Y [M, n]
    int n, mode;
    const float* norm_w;
};
// Y_i = epilogue_i(X W_i) for up to four projections of X [M, K] in one launch
zg_status run_projections(const void* x, long long M, int K, const Proj* pr, int nb, int head_dim,
                          const int32_t* pos, const RopeConsts* rope, float eps, cudaStream_t s) {
    GemmParams g;
    std::memset(&g, 0, sizeof(g));
    if (!dev_ctl(g.ctl)) return ZG_ERR_CUDA;
    if (!make_map_2d(&g.tm_a, x, K, M, gemm_tile_m())) return ZG_ERR_CUDA;
    g.nb = nb;
    g.M = static_cast<int>(M);
    g.K = K;
    g.tiles_m = static_cast<int>((M + gemm_tile_m() - 1) / gemm_tile_m());
    g.head_dim = head_dim;
    g.pos = pos;
    g.eps = eps;
    if (rope) g.rope = *rope;
    long long tn = 0;
    for (int i = 0; i < nb; ++i) {
        if (!make_map_2d(&g.tm_b[i], pr[i].w, pr[i].n, K, 64)) return ZG_ERR_CUDA;
        g.y[i] = pr[i].y;
        g.w[i] = pr[i].norm_w;
        g.n[i] = pr[i].n;
        g.mode[i] = pr[i].mode;
        g.tiles_n[i] = (pr[i].n + gemm_tile_n() - 1) / gemm_tile_n();
        tn += g.tiles_n[i];
    }
    g.tiles = tn * g.tiles_m;
    return launch_gemm(g, s) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

struct LayerWs {
    size_t q, k, v, g, a, total;
};
LayerWs layer_ws(long long B, long long L, long long Hq, long long Hkv, long long d) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    LayerWs w;
    const size_t tq = static_cast<size_t>(B * L * Hq * d) * 2, tk = static_cast<size_t>(B * L * Hkv * d) * 2;
    w.q = 0;
    w.k = w.q + up(tq);
    w.v = w.k + up(tk);
    w.g = w.v + up(tk);
    w.a = w.g + up(tq);
    w.total = w.a + up(tq);
    return w;
}
}  // namespace

zg_status zg_linear(const zg_bf16* x, const zg_bf16* w, zg_bf16* y, int64_t M, int N, int K, zg_stream stream) {
    if (!x || !w || !y) return ZG_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return ZG_ERR_ALIGN;
    if (M < 0 || N <= 0 || K <= 0 || N % 8 || K % 8) return ZG_ERR_SHAPE;
    if (M >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    if (M == 0) return ZG_OK;
    const Proj pr{w, y, N, 0, nullptr};
    return run_projections(x, M, K, &pr, 1, 0, nullptr, nullptr, 0.f, reinterpret_cast<cudaStream_t>(stream));
}

size_t zg_gated_swa_layer_workspace_bytes(int B, int L, int Hq, int Hkv, int d) {
    if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return 0;
    return layer_ws(B, L, Hq, Hkv, d).total;
}

zg_status zg_gated_swa_layer(const zg_bf16* h, const zg_bf16* w_q, const zg_bf16* w_k, const zg_bf16* w_v,
                             const zg_bf16* w_g, const zg_bf16* w_o, const int32_t* pos, const float* wq,
                             const float* wk, zg_bf16* y, int B, int L, int hidden, int Hq, int Hkv, int d,
                             int window, int rotary_dim, double theta, float eps, void* workspace,
                             size_t workspace_bytes, zg_stream stream) {
    if (!h || !w_q || !w_k || !w_v || !w_g || !w_o || !y) return ZG_ERR_NULL;
    if (!aligned16(h) || !aligned16(w_q) || !aligned16(w_k) || !aligned16(w_v) || !aligned16(w_g) ||
        !aligned16(w_o) || !aligned16(y))
        return ZG_ERR_ALIGN;
    if (hidden <= 0 || hidden % 8) return ZG_ERR_SHAPE;  // rows of 16-byte multiples for the GEMMs
    // the attention's own checks, on stand-in pointers (the real q/k/v/gate live in the workspace)
    const zg_bf16* stand_in = h;
    zg_status st = check_prefill(stand_in, stand_in, stand_in, stand_in, true, pos, wq, wk, y, B, L, Hq, Hkv, d,
                                 rotary_dim, theta, eps);
    if (st != ZG_OK) return st;
    if (window < 1) return ZG_ERR_SHAPE;
    const int G = Hq / Hkv;
    if ((d != 64 && d != 128) || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) || window > 128 ||
        Hkv > 65535 || rotary_dim > 64)  // the fused epilogue rotates inside a head's first 64 columns
        return ZG_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return ZG_OK;
    const long long M = static_cast<long long>(B) * L;
    if (M >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    const LayerWs w = layer_ws(B, L, Hq, Hkv, d);
    if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return ZG_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void *qh = base + w.q, *kh = base + w.k, *v = base + w.v, *sg = base + w.g, *a = base + w.a;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    RopeConsts rc;
    if (!rope_consts(rc, rotary_dim, theta)) return ZG_ERR_SHAPE;
    // 1. the four input projections in one launch, h read once: q_hat, k_hat (fp16, RMSNorm and RoPE
    //    from the fp32 accumulator), v (bf16), sigmoid(g) (bf16)
    const Proj in[4] = {{w_q, qh, Hq * d, 1, wq}, {w_k, kh, Hkv * d, 1, wk}, {w_v, v, Hkv * d, 0, nullptr},
                        {w_g, sg, Hq * d, 2, nullptr}};
    st = run_projections(h, M, hidden, in, 4, d, pos, &rc, eps, s);
    if (st != ZG_OK) return st;
    // 2. the windowed attention on the pre-normalised inputs (no Q / K transform, no sigmoid)
    const int T = 128 / G;
    const long long n_lt = (L + T - 1) / T;
    if (n_lt * Hkv * B >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    PrefillParams p;
    std::memset(&p, 0, sizeof(p));
    if (!dev_ctl(p.ctl)) return ZG_ERR_CUDA;
    const int NK = swa_kv_box_rows(G);
    if (!make_map(&p.tm_q, qh, d, Hq, L, B, G, T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
        !make_map(&p.tm_gate, sg, d, Hq, L, B, G, T) || !make_map(&p.tm_out, a, d, Hq, L, B, G, T) ||
        !make_map(&p.tm_k, kh, d, Hkv, L, B, 1, NK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
        !make_map(&p.tm_v, v, d, Hkv, L, B, 1, NK))
        return ZG_ERR_CUDA;
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = window;
    p.n_ltiles = static_cast<int>(n_lt);
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    p.rope = rc;
    p.pre = 1;
    if (launch_swa_prefill(p, d, s) != cudaSuccess) return ZG_ERR_CUDA;
    // 3. o_proj
    const Proj out{w_o, y, hidden, 0, nullptr};
    return run_projections(a, M, Hq * d, &out, 1, 0, nullptr, nullptr, 0.f, s);
}

// ---------------------------------------------------------------- attention backward
size_t zg_attention_backward_workspace_bytes(int B, int L, int Hq, int Hkv, int d) {
    if (B <= 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || d != 128) return 0;
    return backward_workspace_bytes(B, L, Hq, Hkv);
}

zg_status zg_attention_backward(const zg_bf16* q, const zg_bf16* k, const zg_bf16* v, const zg_bf16* gate,
                                const int32_t* pos, const float* wq, const float* wk, const zg_bf16* dout, float* dq,
                                float* dk, float* dv, float* dgate, int B, int L, int Hq, int Hkv, int d, int window,
                                int rotary_dim, double theta, float eps, void* workspace, size_t workspace_bytes,
                                zg_stream stream) {
    const bool gated = gate != nullptr;
    if (!q || !k || !v || !pos || !wq || !wk || !dout || !dq || !dk || !dv || (gated && !dgate)) return ZG_ERR_NULL;
    if (!gated && dgate) return ZG_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (gated && !aligned16(gate)) || !aligned16(pos) ||
        !aligned16(wq) || !aligned16(wk) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (gated && !aligned16(dgate)))
        return ZG_ERR_ALIGN;
    if (B < 0 || L < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return ZG_ERR_SHAPE;
    if (rotary_dim < 0 || rotary_dim > d || (rotary_dim & 1) || !(theta > 0.0) || !(eps >= 0.0f)) return ZG_ERR_SHAPE;
    if (d != 128) return ZG_ERR_UNSUPPORTED;
    if (B == 0 || L == 0) return ZG_OK;
    if (static_cast<long long>(B) * L * (Hq + Hkv) / 8 >= (1ll << 31)) return ZG_ERR_UNSUPPORTED;
    const size_t need = backward_workspace_bytes(B, L, Hq, Hkv);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return ZG_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the global layer (every earlier key, no gate) on the tensor cores too
    const bool global_tc = !gated && (window <= 0 || window >= L) && backward_tc_global_supports(d, Hq, Hkv);
    const bool tc = (backward_tc_supports(d, Hq, Hkv, window) || global_tc) && Hkv <= 65535 &&
                    static_cast<long long>(B) * Hkv * ((L + 31) / 32) < (1ll << 31) &&
                    static_cast<long long>(B) * L * (Hq + Hkv) < (1ll << 31);
    if (tc) {
        // tensor-core path (the ZGCM-1 local-layer shape)
        BackwardTcParams t;
        std::memset(&t, 0, sizeof(t));
        if (!dev_ctl(t.ctl)) return ZG_ERR_CUDA;
        const size_t rq = static_cast<size_t>(B) * L * Hq * d, rk = static_cast<size_t>(B) * L * Hkv * d;
        uint8_t* w8 = static_cast<uint8_t*>(workspace);
        t.qh = reinterpret_cast<__nv_bfloat16*>(w8);
        t.da = reinterpret_cast<__nv_bfloat16*>(w8 + rq * 2);
        t.kh = reinterpret_cast<__nv_bfloat16*>(w8 + rq * 4);
        t.stat = reinterpret_cast<float4*>(w8 + rq * 4 + rk * 2);
        const void* da_src = gated ? static_cast<const void*>(t.da) : static_cast<const void*>(dout);
        if (!make_map(&t.tm_qh, t.qh, d, Hq, L, B, 4, 32) || !make_map(&t.tm_da, da_src, d, Hq, L, B, 4, 32) ||
            !make_map(&t.tm_kq, t.kh, d, Hkv, L, B, 1, 160) || !make_map(&t.tm_vq, v, d, Hkv, L, B, 1, 160) ||
            !make_map(&t.tm_kk, t.kh, d, Hkv, L, B, 1, 128) || !make_map(&t.tm_vk, v, d, Hkv, L, B, 1, 128) ||
            !make_map(&t.tm_q, q, d, Hq, L, B, 4, 32) || !make_map(&t.tm_kraw, k, d, Hkv, L, B, 1, 128) ||
            !make_map_f32(&t.tm_dqf, dq, d, Hq, L, B, 4, 32) || !make_map_f32(&t.tm_dkf, dk, d, Hkv, L, B, 1, 128) ||
            !make_map_f32(&t.tm_dvf, dv, d, Hkv, L, B, 1, 128))
            return ZG_ERR_CUDA;
        if (gated && (!make_map(&t.tm_gate, gate, d, Hq, L, B, 4, 32) || !make_map(&t.tm_dout, dout, d, Hq, L, B, 4, 32) ||
                      !make_map_f32(&t.tm_dg, dgate, d, Hq, L, B, 4, 32)))
            return ZG_ERR_CUDA;
        t.q = reinterpret_cast<const __nv_bfloat16*>(q);
        t.k = reinterpret_cast<const __nv_bfloat16*>(k);
        t.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
        t.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
        t.pos = pos;
        t.wq = wq;
        t.wk = wk;
        t.dq = dq;
        t.dk = dk;
        t.dv = dv;
        t.dgate = dgate;
        t.B = B;
        t.L = L;
        t.Hq = Hq;
        t.Hkv = Hkv;
        t.global = global_tc ? 1 : 0;
        t.fold = !global_tc && rotary_dim <= 64 ? 1 : 0;
        t.window = global_tc ? L : window;
        t.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
        t.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
        t.eps = eps;
        if (!rope_consts(t.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
        return launch_backward_tc(t, s) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
    }
    BackwardParams p;
    std::memset(&p, 0, sizeof(p));
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(k);
    p.v = reinterpret_cast<const __nv_bfloat16*>(v);
    p.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
    p.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dgate = dgate;
    const size_t rq = static_cast<size_t>(B) * L * Hq * d, rk = static_cast<size_t>(B) * L * Hkv * d;
    float* f = static_cast<float*>(workspace);
    p.qh = f;
    p.da = f + rq;
    p.dqh = f + 2 * rq;
    p.kh = f + 3 * rq;
    p.dkh = f + 3 * rq + rk;
    p.stat = f + 3 * rq + 2 * rk;
    p.B = B;
    p.L = L;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.window = window > 0 ? window : 0;
    p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    if (!rope_consts(p.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_backward(p, d, s) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

size_t zg_hybrid_decode_workspace_bytes(int NG, int B, int Hq, int d, int64_t S_max) {
    if (NG <= 0 || B <= 0 || Hq <= 0 || d <= 0 || S_max <= 0) return 0;
    return decode_workspace_bytes(NG, B, Hq, d, S_max);
}


// one decode step over bf16 (fp8 = 0) or E4M3 (fp8 = 1) caches
static zg_status hybrid_decode_impl(const zg_bf16* q, const zg_bf16* k_new, const zg_bf16* v_new, const zg_bf16* gate,
                                    const int32_t* pos, const float* wq, const float* wk, const uint8_t* is_global,
                                    void* k_glob, void* v_glob, void* k_ring, void* v_ring, zg_bf16* out, int NL,
                                    int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim,
                                    double theta, float eps, void* workspace, size_t workspace_bytes, int fp8,
                                    float k_scale, float v_scale, zg_stream stream) {
    int NG = 0;
    const zg_status st = (zg_status)hybrid_decode_check(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring,
                                       out, NL, B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, fp8, k_scale,
                                       v_scale, &NG);
    if (st != ZG_OK) return st;
    if (NL == 0 || B == 0) return ZG_OK;
    int NS = 0;
    int glob_layers[kMaxLayers], loc_layers[kMaxLayers];
    NG = 0;
    for (int l = 0; l < NL; ++l) {
        if (is_global[l]) glob_layers[NG++] = l;
        else loc_layers[NS++] = l;
    }
    const size_t need = NG ? decode_workspace_bytes(NG, B, Hq, d, S_max) : 0;
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return ZG_ERR_WORKSPACE;
    const long long nsplit = NG ? (S_max + kDecodeSplitLen - 1) / kDecodeSplitLen : 1;

    DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    if (!dev_ctl(p.ctl)) return ZG_ERR_CUDA;
    const int box_rows = decode_cache_box_rows(d, fp8 != 0);
    if (NG && (!make_cache_map(&p.tm_kg, k_glob, d, S_max, static_cast<long long>(NG) * B * Hkv, fp8, box_rows) ||
               !make_cache_map(&p.tm_vg, v_glob, d, S_max, static_cast<long long>(NG) * B * Hkv, fp8, box_rows)))
        return ZG_ERR_CUDA;
    if (NS && (!make_cache_map(&p.tm_kr, k_ring, d, window, static_cast<long long>(NS) * B * Hkv, fp8, box_rows) ||
               !make_cache_map(&p.tm_vr, v_ring, d, window, static_cast<long long>(NS) * B * Hkv, fp8, box_rows)))
        return ZG_ERR_CUDA;
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
    p.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
    p.gate = reinterpret_cast<const __nv_bfloat16*>(gate);
    p.pos = pos;
    p.wq = wq;
    p.wk = wk;
    p.k_glob = static_cast<__nv_bfloat16*>(k_glob);  // E4M3 bytes when fp8
    p.v_glob = static_cast<__nv_bfloat16*>(v_glob);
    p.k_ring = static_cast<__nv_bfloat16*>(k_ring);
    p.v_ring = static_cast<__nv_bfloat16*>(v_ring);
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    const size_t rows = static_cast<size_t>(NG) * B * Hq * static_cast<size_t>(nsplit);
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = NG ? static_cast<float*>(workspace) + rows * d : nullptr;
    p.NL = NL;
    p.NG = NG;
    p.NS = NS;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.W = window;
    p.S = NG ? S_max : (1ll << 31) - 1;  // local-only stacks: any position >= 0 is valid
    p.split_len = kDecodeSplitLen;
    p.nsplit = static_cast<int>(nsplit);
    for (int i = 0; i < NG; ++i) p.layer_of_global[i] = glob_layers[i];
    for (int i = 0; i < NS; ++i) p.layer_of_local[i] = loc_layers[i];
    p.fp8 = fp8;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.eps = eps;
    if (!rope_consts(p.rope, rotary_dim, theta)) return ZG_ERR_SHAPE;
    return launch_hybrid_decode(p, d, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

zg_status zg_hybrid_decode(const zg_bf16* q, const zg_bf16* k_new, const zg_bf16* v_new, const zg_bf16* gate,
                           const int32_t* pos, const float* wq, const float* wk, const uint8_t* is_global,
                           zg_bf16* k_glob, zg_bf16* v_glob, zg_bf16* k_ring, zg_bf16* v_ring, zg_bf16* out, int NL,
                           int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim, double theta,
                           float eps, void* workspace, size_t workspace_bytes, zg_stream stream) {
    return hybrid_decode_impl(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, out, NL,
                              B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, workspace, workspace_bytes, 0,
                              1.0f, 1.0f, stream);
}

zg_status zg_hybrid_decode_fp8(const zg_bf16* q, const zg_bf16* k_new, const zg_bf16* v_new, const zg_bf16* gate,
                               const int32_t* pos, const float* wq, const float* wk, const uint8_t* is_global,
                               uint8_t* k_glob, uint8_t* v_glob, uint8_t* k_ring, uint8_t* v_ring, zg_bf16* out,
                               int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim,
                               double theta, float eps, float k_scale, float v_scale, void* workspace,
                               size_t workspace_bytes, zg_stream stream) {
    return hybrid_decode_impl(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, out, NL,
                              B, Hq, Hkv, d, S_max, window, rotary_dim, theta, eps, workspace, workspace_bytes, 1,
                              k_scale, v_scale, stream);
}

zg_status zg_device_status(uint32_t* detail) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ZG_ERR_CUDA;
    uint32_t w = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return ZG_ERR_CUDA;
    if (w && cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return ZG_ERR_CUDA;
    if (detail) *detail = w;
    if (!w) return ZG_OK;
    if ((w & 0xFFu) == kErrPosition) return ZG_ERR_POSITION;
    if ((w & 0xFFu) == kErrIndex) return ZG_ERR_DEVICE_INDEX;
    return ZG_ERR_DEVICE_TIMEOUT;
}

zg_status zg_selftest_index_check(zg_stream stream) {
    DevCtl ctl;
    if (!dev_ctl(ctl)) return ZG_ERR_CUDA;
    return launch_index_selftest(ctl, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

int zg_debug_build(void) {
#ifdef ZG_DEBUG
    return 1;
#else
    return 0;
#endif
}

zg_status zg_selftest_bounded_wait(uint64_t limit_ns, zg_stream stream) {
    DevCtl ctl;
    if (!dev_ctl(ctl)) return ZG_ERR_CUDA;
    ctl.wait_limit_ns = limit_ns;
    return launch_wait_selftest(ctl, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ZG_OK : ZG_ERR_CUDA;
}

const char* zg_status_string(int s) {
    switch (s) {
        case ZG_OK: return "ok";
        case ZG_ERR_NULL: return "null pointer";
        case ZG_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ZG_ERR_SHAPE: return "invalid size or parameter";
        case ZG_ERR_UNSUPPORTED: return "shape not supported by the kernels";
        case ZG_ERR_POSITION: return "position outside the cache";
        case ZG_ERR_WORKSPACE: return "workspace missing or too small";
        case ZG_ERR_CUDA: return "CUDA runtime error";
        case ZG_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case ZG_ERR_UNIMPLEMENTED: return "not implemented";
        case ZG_ERR_DEVICE_INDEX: return "device-side index out of range (debug build)";
        default: return "unknown status";
    }
}

}  // extern "C"
