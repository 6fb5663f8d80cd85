/*
 * zg_attn.h -- C ABI of the ZGCM-1 attention hot path for NVIDIA B300 (sm_103a).
 *
 * The operation (sources by page title and section):
 *   "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ"
 *   (architecture): 27 of the 32 layers are gated sliding-window GQA attention
 *   over the most recent 128 tokens, GatedSWA(h) = o_proj(A_SWA(q,k,v) ⊙
 *   σ(g_proj(h))); the other 5 layers (0-indexed 5, 11, 17, 23, 29) are global
 *   causal attention without the gate; q and k get QK RMSNorm and partial RoPE
 *   with rotary ratio 0.33; the decode KV cache keeps 128 tokens for local
 *   layers and the whole sequence for global layers.
 *   "ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for Math and
 *   Agentic Search" (jaehun.me review), section "게이트형 SWA의 동작": a window
 *   of W tokens includes the query token itself; the gate is element-wise.
 *   Same review, section "KV 캐시가 6.4배 줄어드는 이유": 20 KiB of cache per
 *   token for the hybrid stack against 128 KiB for full attention.
 *   hyper.ai summary of arXiv 2609.13356, section "方法": the GatedSWA equation.
 *
 * What every entry point computes, per query token i and query head h, with
 * KV head g = floor(h * Hkv / Hq) and d = head_dim:
 *   q_hat = RoPE(RMSNorm(q[i,h]; wq, eps), pos[i])      k_hat_j likewise (wk)
 *   RMSNorm(x; w, eps) = x * (mean(x^2) + eps)^(-1/2) * w     (over d values)
 *   RoPE: dims [0, r) rotate in pairs (j, j + r/2) by pos * theta^(-2j/r);
 *         dims [r, d) pass through.  r = rotary_dim (even).
 *   A = sum_j softmax_j(q_hat . k_hat_j / sqrt(d)) v[j,g]
 *   SWA:    j in [max(0, i - window + 1), i]   -> out = A * sigmoid(gate)
 *   global: j in [0, i]                        -> out = A
 * Scores, softmax and accumulation run in fp32; for the prefill tensor cores
 * q_hat and k_hat are rounded to fp16 (RMSNorm bounds them far inside its range)
 * and the softmax weights to bf16; out is rounded to bf16.  sigmoid(gate) is
 * evaluated in fp32 without cancellation for negative logits.
 *
 * Conventions for every call:
 *   - All tensors are device memory, row-major and contiguous, owned by the
 *     caller.  bf16 tensors are passed as zg_bf16 (raw bf16 bits).
 *   - Every tensor pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Arguments are checked on the host BEFORE anything is
 *     launched; a failed check returns a negative zg_status and launches
 *     nothing.  ZG_ERR_CUDA reports a launch failure.
 *   - Device-side waits are bounded (ZG_WAIT_LIMIT_NS in the environment,
 *     default 4 s).  A wait that runs out records itself in a device error
 *     word; zg_device_status() synchronises the device and returns
 *     ZG_ERR_DEVICE_TIMEOUT (or ZG_ERR_POSITION for a cache position without a
 *     slot, or ZG_OK) and clears the word.
 *   - Debug build (libzgattn_debug.so, the same sources compiled with ZG_DEBUG):
 *     before every plain global-memory access (TMA copies are bounds-checked by
 *     the hardware) the kernels check the index against the tensor's extent; an
 *     index out of range is skipped and recorded, and zg_device_status() then
 *     returns ZG_ERR_DEVICE_INDEX.  No trap, no fault: the context stays usable.
 *   - The library allocates no device memory in these calls; scratch memory
 *     comes from a caller-provided workspace (global prefill, decode).
 */
#ifndef ZG_ATTN_H
#define ZG_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t zg_bf16;          /* raw bfloat16 bits */
typedef struct CUstream_st *zg_stream; /* same type as cudaStream_t */

typedef enum {
    ZG_OK = 0,
    ZG_ERR_NULL = -1,           /* a required pointer is NULL */
    ZG_ERR_ALIGN = -2,          /* a pointer is not 16-byte aligned */
    ZG_ERR_SHAPE = -3,          /* a size is negative or inconsistent */
    ZG_ERR_UNSUPPORTED = -4,    /* valid, but not a shape the kernels implement */
    ZG_ERR_POSITION = -5,       /* decode position outside the cache */
    ZG_ERR_WORKSPACE = -6,      /* workspace missing or too small */
    ZG_ERR_CUDA = -7,           /* a CUDA runtime call failed */
    ZG_ERR_DEVICE_TIMEOUT = -8, /* a device-side wait gave up */
    ZG_ERR_UNIMPLEMENTED = -9,
    ZG_ERR_DEVICE_INDEX = -10   /* debug build only: a kernel met a global-memory index out of range */
} zg_status;

/*
 * Gated sliding-window GQA attention prefill (the local layers).
 *   q, gate: [B, L, Hq, d] bf16      k, v: [B, L, Hkv, d] bf16
 *   pos: [B, L] int32 RoPE positions (0 <= pos < 2^24)
 *   wq, wk: [d] float32 QK-norm weights (shared by all heads)
 *   out: [B, L, Hq, d] bf16 (written; must not overlap the inputs)
 *   window: keys per query including itself, 1 <= window <= 128
 * Kernel shapes: d in {64, 128}; Hq / Hkv in {1, 2, 4, 8, 16} (a 128-row
 * tensor-core tile packs 128 / G tokens x the G heads of a KV head, so G must
 * divide 128); Hkv <= 65535.
 * B == 0 or L == 0 is a no-op returning ZG_OK.
 */
zg_status zg_swa_prefill(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v, const zg_bf16 *gate,
                         const int32_t *pos, const float *wq, const float *wk, zg_bf16 *out,
                         int B, int L, int Hq, int Hkv, int d, int window, int rotary_dim,
                         double theta, float eps, zg_stream stream);

/* Bytes of device workspace zg_swa_prefill_host needs: two staging slots of
 * chunk_tokens + the key halo (window - 1 rounded up to 128) tokens of every tensor, and the
 * norm weights (0 for invalid sizes). */
size_t zg_swa_prefill_host_workspace_bytes(int B, int Hq, int Hkv, int d, int window, int chunk_tokens);

/*
 * zg_swa_prefill_host -- zg_swa_prefill on HOST buffers, the copies overlapped with the work.
 *   q, k, v, gate, pos, wq, wk, out: HOST pointers with zg_swa_prefill's layouts (out is
 *        written).  Page-locked (pinned) memory lets the copies run asynchronously and overlap;
 *        pageable memory gives the same result without the overlap.
 *   The sequence is processed in chunks of chunk_tokens tokens (every sequence of the batch at
 *   once): chunk c's inputs go to the device (its keys, values and positions with the window's
 *   key halo before it), the prefill kernel runs on it, and its output rows come back, on three
 *   internal streams, so that the copy of chunk c + 1 in, the kernel of chunk c and the copy of
 *   chunk c - 1 out run at the same time.  The halo makes every output identical to one
 *   zg_swa_prefill call over the whole sequence.
 *   workspace: device scratch of at least zg_swa_prefill_host_workspace_bytes() bytes,
 *        16-byte aligned (ZG_ERR_WORKSPACE otherwise); no initialisation.
 *   stream: the work starts after the stream's earlier work and the stream waits for the last
 *        copy back, so a synchronisation of the stream (or the device) completes the call.
 * Errors as zg_swa_prefill (ZG_ERR_SHAPE also for chunk_tokens < 1), plus ZG_ERR_CUDA.
 */
zg_status zg_swa_prefill_host(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v, const zg_bf16 *gate,
                              const int32_t *pos, const float *wq, const float *wk, zg_bf16 *out, int B, int L,
                              int Hq, int Hkv, int d, int window, int rotary_dim, double theta, float eps,
                              int chunk_tokens, void *workspace, size_t workspace_bytes, zg_stream stream);

/* Bytes of workspace zg_global_prefill needs: B * L * Hkv * d * 2 (0 for empty input). */
size_t zg_global_prefill_workspace_bytes(int B, int L, int Hkv, int d);

/*
 * Global (full causal, ungated) GQA attention prefill (the global layers).
 * Same layouts as zg_swa_prefill without gate and window.
 *   workspace: device scratch of at least zg_global_prefill_workspace_bytes()
 *        bytes, 16-byte aligned; it receives the normalised, rotated keys (fp16)
 *        and needs no initialisation.  ZG_ERR_WORKSPACE if missing or too small.
 * Kernel shapes: d in {64, 128}; Hq / Hkv in {1, 2, 4, 8, 16} (as zg_swa_prefill).
 */
zg_status zg_global_prefill(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v,
                            const int32_t *pos, const float *wq, const float *wk, zg_bf16 *out,
                            int B, int L, int Hq, int Hkv, int d, int rotary_dim,
                            double theta, float eps, void *workspace, size_t workspace_bytes,
                            zg_stream stream);

/*
 * Prefill that also leaves the decode caches of its layer behind ("ZGCM-1-7B 完全解説",
 * section "アーキテクチャ": local layers keep the most recent 128 tokens, global layers
 * the whole sequence).  Each call runs the prefill above (same arguments, same output)
 * and then writes, for its layer, the caches zg_hybrid_decode reads:
 *   k cache slot = bf16(RoPE(RMSNorm(k[b,i,g]; wk, eps), pos[b,i]))   (k_hat)
 *   v cache slot = v[b,i,g]
 * zg_swa_prefill_with_cache: k_ring, v_ring are one local layer's rings
 *   [B, Hkv, ring_slots, d] bf16; the last min(L, ring_slots) tokens of every
 *   sequence go to slot pos[b,i] mod ring_slots (ring_slots = the decode window, 128
 *   for ZGCM-1; the last ring_slots positions must differ mod ring_slots, as
 *   consecutive positions do).  Other slots are left untouched.
 * zg_global_prefill_with_cache: k_cache, v_cache are one global layer's caches
 *   [B, Hkv, S_max, d] bf16; every token goes to slot pos[b,i], 0 <= pos < S_max.
 * Head sizes d = 64 and 128 (those of the decode step) are supported, with B <= 65535,
 * L * Hkv < 2^31 and ring_slots < 2^31: ZG_ERR_UNSUPPORTED otherwise.  The cache pointers
 * must be 16-byte aligned and are written in place.
 * A token whose position has no slot (negative, or >= S_max for a global cache) is
 * skipped and recorded on the device: zg_device_status() then returns
 * ZG_ERR_POSITION.  The pages define no interface; these calls follow the cache
 * layout of zg_hybrid_decode.
 */
/*
 * zg_kv_cache_write -- the cache writing of the two calls above on its own: for
 * every sequence b and token i (ring = 1: the last min(L, S) tokens, slot
 * pos[b,i] mod S; ring = 0: every token, slot pos[b,i], 0 <= pos < S) it stores
 * k_hat (bf16) in k_cache and v in v_cache, [B, Hkv, S, d] bf16 each.
 * k, v [B, L, Hkv, d] bf16; pos [B, L] int32; wk [d] float; d = 64 or 128.
 * Errors as for the calls above; positions without a slot are skipped and
 * reported through zg_device_status() as ZG_ERR_POSITION.
 */
zg_status zg_kv_cache_write(const zg_bf16 *k, const zg_bf16 *v, const int32_t *pos, const float *wk,
                            zg_bf16 *k_cache, zg_bf16 *v_cache, int B, int L, int Hkv, int d,
                            int64_t S, int ring, int rotary_dim, double theta, float eps,
                            zg_stream stream);
zg_status zg_swa_prefill_with_cache(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v,
                                    const zg_bf16 *gate, const int32_t *pos, const float *wq,
                                    const float *wk, zg_bf16 *out, int B, int L, int Hq, int Hkv,
                                    int d, int window, int rotary_dim, double theta, float eps,
                                    zg_bf16 *k_ring, zg_bf16 *v_ring, int ring_slots,
                                    zg_stream stream);
zg_status zg_global_prefill_with_cache(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v,
                                       const int32_t *pos, const float *wq, const float *wk,
                                       zg_bf16 *out, int B, int L, int Hq, int Hkv, int d,
                                       int rotary_dim, double theta, float eps, void *workspace,
                                       size_t workspace_bytes, zg_bf16 *k_cache, zg_bf16 *v_cache,
                                       int64_t S_max, zg_stream stream);

/*
 * Bytes of workspace zg_hybrid_decode needs for these sizes (0 when there is
 * no global layer).  NG = number of global layers, S_max = global-cache slots.
 */
size_t zg_hybrid_decode_workspace_bytes(int NG, int B, int Hq, int d, int64_t S_max);

/*
 * One decode step through an NL-layer hybrid stack: every layer gets one new
 * token per sequence.  Layers are independent here (their q/k/v/gate come in
 * precomputed).  Per layer l and sequence b, at position p = pos[b]:
 *   k_hat = RoPE(RMSNorm(k_new; wk[l]), p) is written into the layer's cache
 *   (global layer: slot p of its full cache; local layer: slot p mod W of its
 *   ring) together with v_new, and the new q attends to
 *     global: positions 0..p          -> out = A
 *     local:  positions max(0,p-W+1)..p (min(p+1, W) ring slots)
 *                                      -> out = A * sigmoid(gate)
 * Cache slots hold post-norm, post-RoPE keys and raw values.
 *   q, gate: [NL, B, Hq, d] bf16 (gate rows of global layers are ignored)
 *   k_new, v_new: [NL, B, Hkv, d] bf16
 *   pos: [B] int32 device, 0 <= pos[b] < S_max (positions are not checked on
 *        the host; a position outside the cache makes that sequence's output
 *        zero and records nothing in the cache)
 *   wq, wk: [NL, d] float32
 *   is_global: [NL] uint8, HOST memory; global layers are numbered in order of
 *        appearance into k_glob/v_glob, local layers into k_ring/v_ring
 *   k_glob, v_glob: [NG, B, Hkv, S_max, d] bf16 (updated in place)
 *   k_ring, v_ring: [NS, B, Hkv, W, d] bf16 (updated in place), W = window
 *   out: [NL, B, Hq, d] bf16
 *   workspace: device scratch of at least zg_hybrid_decode_workspace_bytes()
 *        bytes (may be NULL when NG == 0); its contents need no initialisation.
 * Kernel shapes: d = 64 or 128; any GQA ratio 1 <= Hq / Hkv <= 16 (Hq a multiple
 * of Hkv); 1 <= W <= 4096; NL <= 96.  The products run on the warp-level tensor
 * core instruction with fp32 accumulation; q_hat enters them as a bf16 head plus
 * a bf16 tail (about 16 mantissa bits), the softmax weights as bf16 (E4M3
 * caches: q_hat and the weights in fp16).
 */
zg_status zg_hybrid_decode(const zg_bf16 *q, const zg_bf16 *k_new, const zg_bf16 *v_new, const zg_bf16 *gate,
                           const int32_t *pos, const float *wq, const float *wk, const uint8_t *is_global,
                           zg_bf16 *k_glob, zg_bf16 *v_glob, zg_bf16 *k_ring, zg_bf16 *v_ring, zg_bf16 *out,
                           int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim,
                           double theta, float eps, void *workspace, size_t workspace_bytes, zg_stream stream);

/*
 * zg_hybrid_decode_fp8 -- zg_hybrid_decode over E4M3 (FP8) caches.  The pages train
 * with E4M3 in the forward pass ("ZGCM-1-7B 完全解説", gotosocial explainer,
 * section "学習の高速化 — FP8・Muon・TWEOが生む約4.2倍の効率"); here the format holds the decode caches, which are what a decode
 * step reads from HBM, so the bytes per step halve.
 *   k_glob, v_glob [NG, B, Hkv, S_max, d] and k_ring, v_ring [NS, B, Hkv, window, d]:
 *        one byte per element, E4M3 (4 exponent bits, 3 mantissa bits, bias 7, no
 *        infinities), holding e4m3(k_hat * k_scale) and e4m3(v * v_scale).
 *   k_scale, v_scale: finite and > 0 (ZG_ERR_SHAPE otherwise).  QK RMSNorm bounds
 *        |k_hat| by sqrt(d) * max|wk|, so k_scale = 1 keeps keys in range for any
 *        weights below 26; v_scale should map the value range into +-448.
 *   The step writes the new token's slot the same way: round to nearest, saturated
 *   at +-448.  It attends with the new key and value at full precision, and with the
 *   stored ones dequantised (divided by the scales).  Everything else is as
 *   zg_hybrid_decode, including the workspace.
 */
zg_status zg_hybrid_decode_fp8(const zg_bf16 *q, const zg_bf16 *k_new, const zg_bf16 *v_new, const zg_bf16 *gate,
                               const int32_t *pos, const float *wq, const float *wk, const uint8_t *is_global,
                               uint8_t *k_glob, uint8_t *v_glob, uint8_t *k_ring, uint8_t *v_ring, zg_bf16 *out,
                               int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim,
                               double theta, float eps, float k_scale, float v_scale, void *workspace,
                               size_t workspace_bytes, zg_stream stream);

/* zg_kv_cache_write_fp8 -- zg_kv_cache_write into E4M3 caches (one byte per element):
 * e4m3(k_hat * k_scale) and e4m3(v * v_scale), rounded to nearest, saturated at
 * +-448.  Scales finite and > 0 (ZG_ERR_SHAPE otherwise); all else as
 * zg_kv_cache_write. */
zg_status zg_kv_cache_write_fp8(const zg_bf16 *k, const zg_bf16 *v, const int32_t *pos, const float *wk,
                                uint8_t *k_cache, uint8_t *v_cache, int B, int L, int Hkv, int d, int64_t S,
                                int ring, int rotary_dim, double theta, float eps, float k_scale, float v_scale,
                                zg_stream stream);

/* Bytes of workspace zg_global_prefill_fp8 needs: B * Hkv * d * (L + Lp), Lp = L rounded
 * up to a multiple of 16 (0 for empty input). */
size_t zg_global_prefill_fp8_workspace_bytes(int B, int L, int Hkv, int d);

/*
 * zg_global_prefill_fp8 -- zg_global_prefill with E4M3 (FP8) inputs and E4M3 tensor-core
 * products.  The pages run the forward pass's matrix products in E4M3 ("ZGCM-1-7B 完全解説",
 * section "学習の高速化 — FP8・Muon・TWEOが生む約4.2倍の効率"); here both attention
 * products of the global layers take that format (tcgen05 kind::f8f6f4, fp32 accumulation).
 *   q [B, L, Hq, d], k, v [B, L, Hkv, d]: one byte per element, E4M3, holding
 *        e4m3(q * q_scale), e4m3(k * k_scale), e4m3(v * v_scale); the attention is that of
 *        the dequantised inputs (stored / scale).  Scales finite and > 0, else ZG_ERR_SHAPE.
 *   out [B, L, Hq, d] bf16, pos, wq, wk, rotary_dim, theta, eps: as zg_global_prefill.
 *   Rounding: q_hat and k_hat (after RMSNorm and RoPE in fp32) are rounded to E4M3 times a
 *        power-of-two scale that puts their bound sqrt(d) * max|w| just inside +-448 (the
 *        scale is undone exactly in the softmax); the softmax weights P are rounded to
 *        E4M3 (they are at most 2^8 there) and the row sums add the rounded weights (16 per
 *        fp16 lane, then fp32: relative rounding <= 9 * 2^-11); V enters as stored.  Expect a relative error of a few per cent on the
 *        output (three mantissa bits per operand), not the bf16 path's 1e-2.
 *   workspace: device scratch of at least zg_global_prefill_fp8_workspace_bytes() bytes,
 *        16-byte aligned, no initialisation; it receives k_hat in E4M3 and V transposed
 *        to [B, Hkv, d, Lp] so that both operands of both products are K-major.
 * Kernel shapes: d = 128 (one 128-byte row per head vector); Hq / Hkv in {1, 2, 4, 8, 16};
 * ZG_ERR_UNSUPPORTED otherwise.  B == 0 or L == 0 is a no-op returning ZG_OK.
 */
zg_status zg_global_prefill_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, const int32_t *pos,
                                const float *wq, const float *wk, zg_bf16 *out, int B, int L, int Hq, int Hkv,
                                int d, int rotary_dim, double theta, float eps, float q_scale, float k_scale,
                                float v_scale, void *workspace, size_t workspace_bytes, zg_stream stream);

/*
 * zg_swa_prefill_fp8 -- the gated sliding-window prefill (zg_swa_prefill's operation) with E4M3
 * inputs and E4M3 tensor-core products, on the pipeline of zg_global_prefill_fp8 (one persistent
 * CTA per SM walking pairs of query tiles): each query tile visits only the 128-key blocks that
 * meet its queries' windows, masks both window edges, and multiplies by sigmoid(gate) before the
 * bf16 store; sigmoid(gate) is evaluated in fp32 and rounded to bf16 (2^-9 relative at every
 * magnitude) first.
 *   q, k, v: E4M3 as in zg_global_prefill_fp8 (scales likewise); gate [B, L, Hq, d] bf16 logits
 *        (required: ZG_ERR_NULL if missing); window >= 1 (keys i - window + 1 .. i; ZG_ERR_SHAPE
 *        otherwise; no upper bound: a window of L or more is the global layer with a gate).
 *   workspace: the same size and use as zg_global_prefill_fp8's
 *        (zg_global_prefill_fp8_workspace_bytes).
 *   Rounding and expected error as zg_global_prefill_fp8.
 * Kernel shapes: d = 128; Hq / Hkv in {1, 2, 4, 8, 16}; ZG_ERR_UNSUPPORTED otherwise.
 * B == 0 or L == 0 is a no-op returning ZG_OK.
 */
zg_status zg_swa_prefill_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, const zg_bf16 *gate,
                             const int32_t *pos, const float *wq, const float *wk, zg_bf16 *out, int B, int L,
                             int Hq, int Hkv, int d, int window, int rotary_dim, double theta, float eps,
                             float q_scale, float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
                             zg_stream stream);

/*
 * zg_hybrid_decode_noalloc -- the same decode step as zg_hybrid_decode, for
 * callers that cannot allocate device memory (no counterpart in the paper: it
 * exists for how the library is called, not for what it computes).
 *
 * Some callers cannot call cudaMalloc: a plugin inside a host application whose
 * memory manager owns every device allocation and lends none to plugins, or a
 * serving loop that must not allocate while answering requests.  They still own
 * and pass every input and output; only the split-K scratch moves into a fixed
 * array of ZG_NOALLOC_SCRATCH_BYTES compiled into the library, which each GPU
 * that loads the library holds until the process exits.  This call allocates
 * nothing.
 *   - Arguments, layouts and results are those of zg_hybrid_decode.
 *   - Sizes whose scratch need (zg_hybrid_decode_workspace_bytes) exceeds
 *     ZG_NOALLOC_SCRATCH_BYTES are rejected with ZG_ERR_WORKSPACE before any
 *     launch.  64 MiB covers, e.g., 5 global layers x 8 sequences x 32 query
 *     heads with 256K-slot caches (42.6 MB).
 *   - The first call in a CUDA context looks up the array's device address in
 *     that context (the device must be current) and keeps it for the context;
 *     a new context on the same device (after cudaDeviceReset, for instance)
 *     gets its own lookup on its first call.  Make the first call of a context
 *     before any stream capture begins.
 *   - Argument errors are reported with the same status as zg_hybrid_decode
 *     would give, before the scratch size is considered.
 *   - All calls share the one array, which keeps the last call's contents; no
 *     clearing is needed between calls, but calls whose kernels overlap on the
 *     GPU (unordered streams) race on it.
 */
#define ZG_NOALLOC_SCRATCH_BYTES (64u << 20)
zg_status zg_hybrid_decode_noalloc(const zg_bf16 *q, const zg_bf16 *k_new, const zg_bf16 *v_new, const zg_bf16 *gate,
                                   const int32_t *pos, const float *wq, const float *wk, const uint8_t *is_global,
                                   zg_bf16 *k_glob, zg_bf16 *v_glob, zg_bf16 *k_ring, zg_bf16 *v_ring, zg_bf16 *out,
                                   int NL, int B, int Hq, int Hkv, int d, int64_t S_max, int window, int rotary_dim,
                                   double theta, float eps, zg_stream stream);

/*
 * A whole gated sliding-window attention layer from the hidden states ("ZGCM-1-7B
 * 完全解説", section "アーキテクチャ"; hyper.ai summary of arXiv 2609.13356, section
 * "方法"): y = o_proj(A_SWA(q, k, v) ⊙ σ(g_proj(h))), with q, k, v and the gate
 * logits projected in parallel from the normalised hidden state h:
 *   q = h W_q, k = h W_k, v = h W_v, g = h W_g;  a = A_SWA(q, k, v) ⊙ σ(g)
 *   (QK RMSNorm with wq / wk and partial RoPE as zg_swa_prefill);  y = a W_o.
 * h [B, L, hidden] bf16; W_q, W_g [hidden, Hq*d], W_k, W_v [hidden, Hkv*d],
 * W_o [Hq*d, hidden], all bf16 row-major with the input dimension first (y = x W);
 * y [B, L, hidden] bf16.  All on the library's own tensor-core kernels, in three
 * launches: the four input projections in one GEMM (h read once) whose epilogues
 * apply RMSNorm + RoPE to q and k straight from the fp32 accumulator (q_hat, k_hat
 * stored fp16), and sigmoid to g (stored bf16; v stored bf16); the windowed
 * attention on those pre-normalised tensors; o_proj (a rounded to bf16).
 * hidden must be a multiple of 8; rotary_dim <= 64; other shape limits as
 * zg_swa_prefill.
 *   workspace: device scratch of at least zg_gated_swa_layer_workspace_bytes()
 *        bytes, 16-byte aligned (q_hat, k_hat, v, sigmoid(g), a);
 *        ZG_ERR_WORKSPACE if missing or too small.
 */
size_t zg_gated_swa_layer_workspace_bytes(int B, int L, int Hq, int Hkv, int d);
zg_status zg_gated_swa_layer(const zg_bf16 *h, const zg_bf16 *w_q, const zg_bf16 *w_k,
                             const zg_bf16 *w_v, const zg_bf16 *w_g, const zg_bf16 *w_o,
                             const int32_t *pos, const float *wq, const float *wk, zg_bf16 *y,
                             int B, int L, int hidden, int Hq, int Hkv, int d, int window,
                             int rotary_dim, double theta, float eps, void *workspace,
                             size_t workspace_bytes, zg_stream stream);

/*
 * y = x W on the library's tensor-core GEMM (the layer's projections): x [M, K],
 * W [K, N], y [M, N], bf16 row-major, fp32 accumulation, y rounded to bf16.
 * N and K multiples of 8 (16-byte rows); M < 2^31.  The pages' model uses it for
 * o_proj (hyper.ai summary of arXiv 2609.13356, section "方法").
 */
zg_status zg_linear(const zg_bf16 *x, const zg_bf16 *w, zg_bf16 *y, int64_t M, int N, int K, zg_stream stream);

/* Gradients of the attention prefill: the backward pass of zg_swa_prefill (gate
 * given, window >= 1) or of zg_global_prefill (gate NULL, window <= 0), the
 * training workload the pages run at 4K ("ZGCM-1-7B 完全解説", gotosocial
 * explainer, section "アーキテクチャ", for the forward it differentiates).
 * With q_hat = RoPE(RMSNorm(q; wq, eps), pos), k_hat likewise, p_ij the softmax
 * over the window of q_hat_i . k_hat_j / sqrt(d), A_i = sum_j p_ij v_j and
 * out_i = A_i * sigmoid(gate_i) (out_i = A_i without a gate), it returns the
 * gradients of sum(out * dout) with respect to q, k, v and gate.  The gradients
 * of the RMSNorm weights wq, wk are not computed.
 *   q, gate, dout: [B, L, Hq, d] bf16;  k, v: [B, L, Hkv, d] bf16;  pos [B, L]
 *        int32;  wq, wk [d] fp32 — the forward's own inputs, layouts as there.
 *   window: keys i - window < j <= i; <= 0 means every j <= i.  Any window
 *        and either gate setting may be combined.
 *   dq, dgate: [B, L, Hq, d] fp32;  dk, dv: [B, L, Hkv, d] fp32, written in full
 *        (not accumulated).  dgate must be NULL exactly when gate is.
 *   d must be 128 (ZG_ERR_UNSUPPORTED otherwise); Hq a multiple of Hkv.
 *   Nothing of the forward is reused: scores are recomputed.  The ZGCM-1 local
 *   layer shape (d = 128, Hq = 4 Hkv, 1 <= window <= 128) runs on the tensor cores
 *   with bf16 operands (q_hat, k_hat, dA, P, dS) and fp32 accumulation; every other
 *   shape (the global layer included) runs in fp32 on the CUDA cores.
 *   All pointers device memory, 16-byte aligned, owned by the caller.
 *   workspace: at least zg_attention_backward_workspace_bytes() bytes, 16-byte
 *        aligned (fp32 q_hat, k_hat, dA, dq_hat, dk_hat and three floats per
 *        query row); ZG_ERR_WORKSPACE if missing or too small.
 */
size_t zg_attention_backward_workspace_bytes(int B, int L, int Hq, int Hkv, int d);
zg_status zg_attention_backward(const zg_bf16 *q, const zg_bf16 *k, const zg_bf16 *v,
                                const zg_bf16 *gate, const int32_t *pos, const float *wq,
                                const float *wk, const zg_bf16 *dout, float *dq, float *dk,
                                float *dv, float *dgate, int B, int L, int Hq, int Hkv, int d,
                                int window, int rotary_dim, double theta, float eps,
                                void *workspace, size_t workspace_bytes, zg_stream stream);

/* Synchronise the current device, return ZG_ERR_DEVICE_TIMEOUT if a device wait
 * gave up since the last call (and clear that record), ZG_ERR_CUDA if the
 * device reports an error, else ZG_OK.  *detail (may be NULL) receives the raw
 * record: (site << 8) | code. */
zg_status zg_device_status(uint32_t *detail);

/* Launch a kernel whose only work is a bounded wait on a barrier that nothing
 * completes, with the given limit in ns; used to test the timeout path.  The
 * caller then reads the outcome with zg_device_status(). */
zg_status zg_selftest_bounded_wait(uint64_t limit_ns, zg_stream stream);

/* Launch a kernel that asks the debug build's index check about an index one past
 * the end of a range, while the access it guards stays in range.  Debug build:
 * zg_device_status() afterwards returns ZG_ERR_DEVICE_INDEX (site 98); normal
 * build: ZG_OK.  Used to test the debug build's error path without a fault. */
zg_status zg_selftest_index_check(zg_stream stream);

/* 1 for the debug build (libzgattn_debug.so, compiled with ZG_DEBUG), else 0. */
int zg_debug_build(void);

/* Static text for a status code. */
const char *zg_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* ZG_ATTN_H */
