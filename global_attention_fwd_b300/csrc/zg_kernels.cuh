// zg_kernels.cuh -- parameter blocks and launch entry points shared by the
// CUDA kernels and the C-ABI layer of the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include <cuda_fp16.h>

#include "zg_ptx.cuh"

namespace zg {

constexpr int kMaxRotHalf = 64;  // rotary_dim / 2 <= head_dim / 2 <= 64

// Per-call RoPE constants computed on the host in double precision:
// inverse frequency theta^(-2j/r) split into a float head and a float tail so the
// device can form pos * f to ~2^-40 relative before reducing it modulo 2*pi.
struct RopeConsts {
    int half;  // rotary_dim / 2
    float f_hi[kMaxRotHalf];
    float f_lo[kMaxRotHalf];
};

// ---------------------------------------------------------------- prefill
struct PrefillParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_gate, tm_out;  // 4-D maps {d, heads, L, B}
    CUtensorMap tm_kh;                               // global prefill: fp16 k_hat workspace
    const void* k_raw;                               // global prefill: raw keys [B, L, Hkv, d] (bf16 or E4M3)
    void* khat;                                      // global prefill: k_hat workspace (fp16, or E4M3)
    const int32_t* pos;                              // [B, L]
    const float* wq;                                 // [d]
    const float* wk;                                 // [d]
    int B, L, Hq, Hkv, window;
    int n_ltiles;      // query tiles along L per (b, kv head)
    int pre;           // SWA: q, k already q_hat, k_hat (fp16) and gate already sigmoid(g) (bf16)
    int swa;           // E4M3 path: the gated sliding-window layer (window, gate map tm_gate) on the global pipeline
    // global prefill over E4M3 inputs: q, k, v hold e4m3(x * scale); these undo the scales
    int fp8;
    const void* v_raw;                               // E4M3 values [B, L, Hkv, d] (transposed by the pre-pass)
    CUtensorMap tm_vt;                               // V^T workspace {Lp, d, Hkv, B}
    uint8_t* vt_ws;                                  // V^T workspace [B, Hkv, d, Lp] (E4M3)
    int vt_lp;                                       // Lp: L rounded up to 16 (16-byte rows)
    float in_dequant_q, in_dequant_k, in_dequant_v;  // 1 / scale of each input
    float scale_log2;  // log2(e) / sqrt(d)
    float eps;
    RopeConsts rope;
    DevCtl ctl;
};

cudaError_t launch_swa_prefill(const PrefillParams& p, int d, cudaStream_t s);
int swa_kv_box_rows(int G);  // rows of the K/V TMA box the SWA kernel for GQA ratio G expects
bool swa2_supports(int d, int G);
cudaError_t launch_swa2_prefill(const PrefillParams& p, int d, cudaStream_t s);
cudaError_t launch_global_prefill(const PrefillParams& p, int d, cudaStream_t s);
bool global_supports(int d, int G);  // head sizes and GQA ratios the global prefill implements
int global_q_tile_tokens(int G);     // tokens of one 128-row query tile (128 / G)

// ---------------------------------------------------------------- decode
struct DecodeParams {
    CUtensorMap tm_kg, tm_vg;    // 3-D maps {d, S, NG*B*Hkv} over the global caches (bf16 or E4M3 bytes)
    CUtensorMap tm_kr, tm_vr;    // 3-D maps {d, W, NS*B*Hkv} over the rings
    const __nv_bfloat16* q;      // [NL, B, Hq, d]
    const __nv_bfloat16* k_new;  // [NL, B, Hkv, d]
    const __nv_bfloat16* v_new;  // [NL, B, Hkv, d]
    const __nv_bfloat16* gate;   // [NL, B, Hq, d]
    const int32_t* pos;          // [B]
    const float* wq;             // [NL, d]
    const float* wk;             // [NL, d]
    __nv_bfloat16* k_glob;       // [NG, B, Hkv, S, d]
    __nv_bfloat16* v_glob;
    __nv_bfloat16* k_ring;       // [NS, B, Hkv, W, d]
    __nv_bfloat16* v_ring;
    __nv_bfloat16* out;          // [NL, B, Hq, d]
    float* ws_o;                 // [NG, B, Hq, nsplit, d] partial outputs
    float* ws_ml;                // [NG, B, Hq, nsplit, 2] partial (max, sum)
    int NL, NG, NS, B, Hq, Hkv, W;
    long long S;
    int split_len;  // keys per split of a global layer
    int nsplit;     // splits per (global layer, b, kv head)
    int layer_of_global[96];  // global-layer index -> layer
    int layer_of_local[96];   // local-layer index -> layer
    int fp8;                  // caches hold E4M3 bytes: e4m3(k_hat * k_scale), e4m3(v * v_scale)
    float k_scale, v_scale;
    float scale_log2;
    float eps;
    RopeConsts rope;
    DevCtl ctl;
};

constexpr int kMaxLayers = 96;
constexpr int kDecodeSplitLen = 8192;  // keys of a global cache per split

cudaError_t launch_hybrid_decode(const DecodeParams& p, int d, cudaStream_t s);
// the host argument checks of one decode step (all but the workspace's); *ng = global layers
int hybrid_decode_check(const void* q, const void* k_new, const void* v_new, const void* gate, const void* pos,
                        const void* wq, const void* wk, const uint8_t* is_global, const void* k_glob,
                        const void* v_glob, const void* k_ring, const void* v_ring, const void* out, int NL, int B,
                        int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim, double theta, float eps,
                        int fp8, float k_scale, float v_scale, int* ng);
size_t decode_workspace_bytes(int NG, int B, int Hq, int d, long long S);
bool decode_supports(int d, int G);          // head sizes and GQA ratios the decode kernels implement
int decode_cache_box_rows(int d, bool fp8);  // cache rows per TMA box of one decode stage

// ---------------------------------------------------------------- decode caches from a prefill
struct CacheParams {
    const __nv_bfloat16* k;  // [B, L, Hkv, d]
    const __nv_bfloat16* v;  // [B, L, Hkv, d]
    const int32_t* pos;      // [B, L]
    const float* wk;         // [d]
    __nv_bfloat16* cache_k;  // [B, Hkv, S, d]: k_hat
    __nv_bfloat16* cache_v;  // [B, Hkv, S, d]: v
    int B, L, Hkv;
    long long S;  // slots: S_max of a global cache, or the ring size
    int ring;     // 1: ring (slot = pos mod S, last min(L, S) tokens); 0: slot = pos
    int i0;       // first token written
    int fp8;      // E4M3 caches: e4m3(k_hat * k_scale), e4m3(v * v_scale)
    float k_scale, v_scale;
    float eps;
    RopeConsts rope;
    DevCtl ctl;
};

cudaError_t launch_kv_cache(const CacheParams& p, int d, cudaStream_t s);

// ---------------------------------------------------------------- attention backward (gated SWA or global)
struct BackwardParams {
    const __nv_bfloat16* q;     // [B, L, Hq, d]
    const __nv_bfloat16* k;     // [B, L, Hkv, d]
    const __nv_bfloat16* v;     // [B, L, Hkv, d]
    const __nv_bfloat16* gate;  // [B, L, Hq, d] or null (no gate)
    const __nv_bfloat16* dout;  // [B, L, Hq, d]
    const int32_t* pos;         // [B, L]
    const float* wq;            // [d]
    const float* wk;            // [d]
    float* dq;                  // [B, L, Hq, d]
    float* dk;                  // [B, L, Hkv, d]
    float* dv;                  // [B, L, Hkv, d]
    float* dgate;               // [B, L, Hq, d] (only with a gate)
    // workspace regions (fp32)
    float* qh;    // [B, L, Hq, d]   q_hat
    float* kh;    // [B, L, Hkv, d]  k_hat
    float* da;    // [B, L, Hq, d]   dA
    float* dqh;   // [B, L, Hq, d]   dq_hat
    float* dkh;   // [B, L, Hkv, d]  dk_hat
    float* stat;  // [B, L, Hq, 3]   row max, 1 / row sum, D = dA . A
    int B, L, Hq, Hkv;
    int window;   // <= 0: every earlier key (global layer)
    float scale;  // 1 / sqrt(d)
    float eps;
    RopeConsts rope;
};

size_t backward_workspace_bytes(int B, int L, int Hq, int Hkv);
// tensor-core path of the same gradients: d = 128, Hq = 4 Hkv, 1 <= window <= 128
struct BackwardTcParams {
    CUtensorMap tm_qh, tm_da;  // q_hat, dA workspace (bf16 [B, L, Hq, d]): box {64, 4 heads, 32 tokens}
    CUtensorMap tm_kq, tm_vq;  // k_hat workspace, v: box {64, 1, 160 tokens}
    CUtensorMap tm_kk, tm_vk;  // k_hat workspace, v: box {64, 1, 128 tokens}
    CUtensorMap tm_q, tm_gate, tm_dout;  // raw q, gate, dout: box {64, 4 heads, 32 tokens}
    CUtensorMap tm_kraw;                 // raw k: box {64, 1, 128 tokens}
    CUtensorMap tm_dg, tm_dqf;           // dgate, dq (fp32): box {32, 4 heads, 32 tokens}, stores
    CUtensorMap tm_dkf, tm_dvf;          // dk, dv (fp32): box {32, 1, 128 tokens}, stores
    const __nv_bfloat16* q;     // raw inputs (RMSNorm backward, dA)
    const __nv_bfloat16* k;
    const __nv_bfloat16* gate;  // or null
    const __nv_bfloat16* dout;
    const int32_t* pos;
    const float* wq;
    const float* wk;
    float* dq;
    float* dk;
    float* dv;
    float* dgate;
    __nv_bfloat16* qh;   // workspace: q_hat [B, L, Hq, d]
    __nv_bfloat16* kh;   // workspace: k_hat [B, L, Hkv, d]
    __nv_bfloat16* da;   // workspace: dA [B, L, Hq, d] (gated layers; dout itself otherwise)
    float4* stat;        // workspace: per query row (max of the log2-scaled scores, 1 / row sum, D, 0)
    int B, L, Hq, Hkv, window;
    int global;  // 1: the global layer (every earlier key, no gate; window = L)
    int fold;    // 1: the windowed query pass forms q_hat and dA itself (rotary_dim <= 64); prep does k_hat only
    int prep_first;  // first row (q rows, then k rows) the prep kernel processes
    float scale, scale_log2, eps;
    RopeConsts rope;
    DevCtl ctl;
};
bool backward_tc_supports(int d, int Hq, int Hkv, int window);
bool backward_tc_global_supports(int d, int Hq, int Hkv);
size_t backward_tc_workspace_bytes(int B, int L, int Hq, int Hkv);
cudaError_t launch_backward_tc(const BackwardTcParams& p, cudaStream_t s);

cudaError_t launch_backward(const BackwardParams& p, int d, cudaStream_t s);

// ---------------------------------------------------------------- projections (tcgen05 GEMM, fused epilogues)
// Y_i = epilogue_i(X W_i) for up to four W_i sharing X; row-major bf16 X [M, K], W_i [K, N_i].
// mode 0: bf16(acc); mode 1: fp16(RoPE(RMSNorm(acc per head_dim columns; w_i), pos[row]));
// mode 2: bf16(sigmoid(acc)).  Requires K % 8 == 0, N_i % 8 == 0 (mode 1: N_i % head_dim == 0,
// head_dim in {64, 128}, rope.half <= 32).
struct GemmParams {
    CUtensorMap tm_a;     // X: box {64 (K), 128 rows}, 128-byte swizzle
    CUtensorMap tm_b[4];  // W_i: box {64 (N), 64 (K)}, 128-byte swizzle
    void* y[4];
    const float* w[4];    // RMSNorm weights [head_dim] (mode 1)
    int n[4], mode[4], tiles_n[4];
    int nb, M, K, tiles_m, head_dim;
    long long tiles;
    const int32_t* pos;   // [M] RoPE positions (mode 1)
    float eps;
    RopeConsts rope;
    DevCtl ctl;
};
cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s);
int gemm_tile_m();
int gemm_tile_n();

// bounded-wait self test: waits on a barrier nothing arrives on
cudaError_t launch_wait_selftest(DevCtl ctl, cudaStream_t s);
// index-check self test: records ZG_ERR_DEVICE_INDEX in the debug build, nothing in the normal one
cudaError_t launch_index_selftest(DevCtl ctl, cudaStream_t s);

}  // namespace zg
