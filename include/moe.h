/*
 * moe.h -- C ABI of libmoe.so: routed-MoE feed-forward step with low-bit expert weights on one GB300 (sm_103a).
 *
 * What is computed (pages cited by title and section):
 *   - Routing: "Mixed-precision compression of DeepSeek-V4-Flash" (lumirain.cn), "The recipe": the router is
 *     kept in F16 and every token uses its top-6 of 256 routed experts. Rule: logits = W_r x, top-k by logit
 *     (ties to the lower expert index), weights = softmax over the k chosen logits. Hash routing of the first
 *     layers: "quant surgery" (blog.meowhead.cn), section 4 (tid2eid table, equal weights).
 *   - Expert FFN: y = sum_r w_r * Down_r( SiLU(Gate_r x) * (Up_r x) ); the gate and up mat-vecs are fused and the
 *     down projection accumulates into the output ("quantization" glossary, ds4-learning.pages.dev, section
 *     "Q4_K routed experts").
 *   - Verify of width 1+K: "Mixed-precision compression...", "What compression does not solve" and "Width drift":
 *     several tokens share one sweep of the expert weights, and row t of a wide verify must equal the width-1
 *     decode of token t bit for bit ("Why this is not a host-side patch").
 *   - Speculative acceptance of drafted tokens: "Mixed-precision compression...", "What compression does not
 *     solve" (keep a draft with probability min(1, p/q); on a rejection draw from the normalised max(p - q, 0)).
 *   - Weight formats: "quantization" glossary, sections "MXFP4" (17-byte blocks: one E8M0 exponent, 32 E2M1
 *     codes; e = 0 is zero) and "core principle" (Q2_K, 84 bytes per 256 weights); INT4 group 32 with a BF16
 *     scale: "DeepSeek-V4-Flash-0731-W4A16" model card (alphaneural.io), quantisation scheme.
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers, allocated and owned by the caller. The library allocates nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls are asynchronous on it.
 *   - Every call returns moe_status_t. Argument and shape errors are found on the host before any launch and
 *     nothing is launched then. MOE_ERR_CUDA reports a failed launch (cudaGetLastError).
 *   - Device-side errors (a bounded wait that ran out) are written to a status word inside the caller's
 *     workspace; read it with moe_get_device_status(). After such an error call moe_workspace_init() again.
 *   - The library keeps no mutable global state except a per-process cache of device properties, the one-time
 *     kernel attribute settings (shared-memory sizes: once per process for the decode and prefill kernels, once
 *     per device for the others; one process drives one GPU) and the static scratch of
 *     moe_expert_ffn_decode_static.
 *   - Host-side fault injection for tests: if the environment variable MOE_FAULT names a call
 *     ("pack", "route", "decode", "verify", "route_ffn", "prefill", "encode", "spec", "norm"), that call returns
 *     MOE_ERR_FAULT_INJECTED
 *     without launching anything.
 */
#ifndef BIT_MOE_DECODE_GB300_MOE_H
#define BIT_MOE_DECODE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_FMT_MXFP4 = 1,   /* 17 B per 32 weights: byte 0 = E8M0 e, bytes 1..16 codes; element 2j = high nibble of
                          byte 1+j, element 2j+1 = low nibble; value E2M1[code] * 2^(e-127), e=0 -> 0, e=255 -> NaN */
  MOE_FMT_INT4G32 = 2, /* 18 B per 32 weights: bytes 0..15 two's-complement 4-bit codes (same nibble order),
                          bytes 16..17 bf16 scale (little endian); value q * scale */
  MOE_FMT_Q2K = 3,     /* 84 B per 256 weights: scales[16] (sc = low nibble, m = high nibble, one per 16 weights),
                          qs[64] (weight i = bits 2(i%4)..2(i%4)+1 of qs[i/4]), fp16 d, fp16 dmin;
                          value d*sc*q - dmin*m */
  MOE_FMT_Q8_0 = 4     /* 34 B per 32 weights: bytes 0..1 fp16 d (little endian), bytes 2..33 two's-complement
                          8-bit codes; value d*q. The shared expert's format ("Q8" in the recipe of
                          "Mixed-precision compression of DeepSeek-V4-Flash"; the pages give no layout, this library
                          defines it). DECODE layout only. */
} moe_format_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, bad enum, misaligned pointer */
  MOE_ERR_SHAPE = 2,               /* a size the kernels do not support (see each call) */
  MOE_ERR_UNSUPPORTED_FORMAT = 3,  /* format not available for this call */
  MOE_ERR_UNSUPPORTED_ARCH = 4,    /* current device is not compute capability 10.3 */
  MOE_ERR_WORKSPACE_TOO_SMALL = 5,
  MOE_ERR_CUDA = 6,                /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 7,      /* a bounded device-side wait ran out (see moe_get_device_status) */
  MOE_ERR_FAULT_INJECTED = 8       /* MOE_FAULT named this call */
} moe_status_t;

const char* moe_status_string(moe_status_t s);
int32_t moe_version(void);
/* Returns MOE_OK if the current device is sm_103 (GB300), MOE_ERR_UNSUPPORTED_ARCH otherwise. */
moe_status_t moe_check_device(void);

/* ---------------------------------------------------------------- weights ---------------------------------------- */

typedef enum { MOE_SRC_BLOCKS = 0, MOE_SRC_F32 = 1 } moe_src_t;
/* DECODE: the mat-vec layout of the decode / verify kernels (all formats). TC: the tensor-core tile layout (MXFP4
 * only) read by the prefill grouped GEMM; PREFILL is its older name. */
typedef enum { MOE_LAYOUT_DECODE = 0, MOE_LAYOUT_TC = 1, MOE_LAYOUT_PREFILL = 1 } moe_layout_t;
typedef enum { MOE_MAT_GATE_UP = 0, MOE_MAT_DOWN = 1 } moe_matrix_t;

/* Bytes of `rows` x `k` weights in the canonical block format (blocks run along k, row-major). */
size_t moe_canonical_bytes(moe_format_t fmt, int64_t rows, int64_t k);

/* Bytes of the packed device layout for n_experts experts. GATE_UP holds Gate [I,H] and Up [I,H] of each expert,
 * DOWN holds Down [H,I]. The layout is expert-major with a fixed per-expert stride equal to
 * moe_packed_bytes(fmt, layout, kind, 1, H, I), so experts can be packed in batches at dst + e * stride.
 * The packed layout holds exactly the canonical bytes, permuted (same bits per weight). Returns 0 for an
 * unsupported combination. */
size_t moe_packed_bytes(moe_format_t fmt, moe_layout_t layout, moe_matrix_t kind, int64_t n_experts, int64_t H,
                        int64_t I);

/* GPU encoder: fp32 weights [rows, k] (row-major) -> canonical blocks (moe_canonical_bytes(fmt, rows, k) bytes).
 * MXFP4: per 32 weights e = clamp(k0 + 127, 1, 254) with k0 the smallest integer such that amax <= 6 * 2^k0;
 *        code = nearest E2M1 value of w * 2^(127-e), ties to the even code, sign kept on zero.
 * INT4:  for r in {6/7, 0.9, 0.95, 1.0, 1.05, 1.1}: s = amax*r/7 (amax >= 1e-8), q = clamp(rint(w/s), -8, 7);
 *        keep the first r with the smallest fp32 sum of (w - q*s)^2; scale stored as bf16(s) (the model card's
 *        "FP4 -> INT4 conversion", step 2).
 * Q2_K:  per 16-weight group lo = min(0, min w), s_g = (max w - lo)/3, o_g = -lo; d = fp16(max s_g / 15),
 *        dmin = fp16(max o_g / 15); sc = rint(s_g/d), m = rint(o_g/dmin) clamped to [0,15];
 *        q = clamp(rint((w + dmin*m)/(d*sc)), 0, 3) (the pages give no encoder; this is the library's own).
 * Q8_0:  per 32 weights d = fp16(amax / 127); q = clamp(rint(w / d), -127, 127), q = 0 where d = 0 or w / d is
 *        NaN (the library's own; -128 is never produced).
 * All arithmetic fp32 round-to-nearest-even; bit-identical to the CPU oracle. k must be a multiple of the block
 * size. src and dst device pointers; dst 16-byte aligned is not required. */
moe_status_t moe_encode_blocks(moe_format_t fmt, const float* src, int64_t rows, int64_t k, void* dst, void* stream);

/* Pack weights into the device layout.
 *   kind GATE_UP: src_a = Gate, src_b = Up, each [n_experts, I, H];  kind DOWN: src_a = Down [n_experts, H, I],
 *   src_b unused. With src_kind BLOCKS the sources are canonical blocks, with F32 they are fp32 weights that are
 *   encoded on the fly exactly as moe_encode_blocks does.
 *   dst must be 16-byte aligned and hold moe_packed_bytes(...) bytes.
 * Shapes: H and I multiples of 256 (and of the block size), 256 <= H, I <= 4096.
 * Layout MOE_LAYOUT_TC is MXFP4 only; every run is 8704 contiguous bytes: 8192 bytes of codes (even k in the low
 * nibble) then 512 E8M0 exponents permuted for the tensor cores (byte l*16 + c*4 + b = operand row l + 32c, byte b).
 *   GATE_UP (R = 2I rows in groups of 128 = 64 gate rows then the same 64 up rows, K = H): 128 x 128 tiles in
 *   (row tile, column tile) order, codes [128 rows][64 B], b = 32-block of the tile.
 *   DOWN (R = H, K = I): chunks of 256 rows x 64 columns in (column block k / 64, row pair r / 256) order, codes
 *   [256 rows][32 B]; b = 2 * (128-row half of the chunk) + 32-block of the 64 columns. The 64 columns of a chunk
 *   are the 64 intermediate indices one gate/up tile row produces. */
moe_status_t moe_pack_weights(moe_format_t fmt, moe_src_t src_kind, moe_layout_t layout, moe_matrix_t kind,
                              int64_t n_experts, int64_t H, int64_t I, const void* src_a, const void* src_b,
                              void* dst, size_t dst_bytes, void* stream);

/* One layer's packed experts. */
typedef struct {
  moe_format_t fmt;
  moe_layout_t layout;
  int32_t H;              /* hidden size */
  int32_t I;              /* expert intermediate size */
  int32_t E;              /* number of routed experts */
  const void* gate_up;    /* moe_packed_bytes(fmt, layout, MOE_MAT_GATE_UP, E, H, I) bytes */
  const void* down;       /* moe_packed_bytes(fmt, layout, MOE_MAT_DOWN, E, H, I) bytes */
} moe_layer_t;

/* ---------------------------------------------------------------- routing ---------------------------------------- */

/* Router for T tokens.
 *   Softmax mode (token_ids == NULL): logits[t,e] = sum_h W_r[e,h] * x[t,h] (fp16 x bf16 products, fp32 sums),
 *     idx[t, 0..k) = the k largest logits in decreasing order, ties to the lower expert index,
 *     weights[t, r] = exp(l_r - l_0) / sum_j exp(l_j - l_0) over the k chosen (fp32).
 *     An expert whose logit is NaN or -inf is never chosen (NaN is not ordered). If fewer than k experts remain,
 *     the missing ranks get idx 0x7fffffff and weight 0 (NaN weights when none remains); an FFN call given such
 *     ids, and moe_route_expert_ffn, record MOE_ERR_INVALID_ARG (see the decode call for what y holds then).
 *   Hash mode (token_ids != NULL): idx[t, r] = tid2eid[token_ids[t] * k + r], weights = 1/k.
 * router_w_f16 [E, H] fp16; x_bf16 [T, H] bf16; idx [T, k] int32; weights [T, k] fp32.
 * Limits: 1 <= k <= 8, k <= E <= 1024, H multiple of 256 and <= 8192, T >= 1.
 * Token ids outside [0, V) return MOE_ERR_INVALID_ARG only if checked on the host: they are device data, so
 * the kernel clamps nothing and the caller must pass valid ids. */
moe_status_t moe_route_topk(const void* router_w_f16, const void* x_bf16, int32_t T, int32_t H, int32_t E,
                            int32_t k, const int32_t* token_ids, const int32_t* tid2eid, int32_t V, int32_t* idx,
                            float* weights, void* stream);

/* ---------------------------------------------------------------- expert FFN ------------------------------------- */

/* Workspace (device scratch owned by the caller) for decode / verify of up to T_max tokens with top-k.
 * It must be zeroed once with moe_workspace_init() before first use; the kernels leave it zeroed. */
size_t moe_workspace_bytes(const moe_layer_t* layer, int32_t T_max, int32_t k);
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);
/* Synchronises `stream`, returns the device status word (MOE_OK, MOE_ERR_DEVICE_TIMEOUT, or MOE_ERR_INVALID_ARG for
 * an expert id outside [0, E)) and clears it. */
moe_status_t moe_get_device_status(void* ws, void* stream);

/* Decode, one token: y[H] (=, or += if accumulate) sum_r w[r] * FFN_{idx[r]}(x).
 *   x_bf16 [H] bf16; idx [k] int32 (expert ids < E); w [k] fp32; y [H] fp32; y_bf16 [H] bf16 or NULL
 *   (round-to-nearest-even copy of y). Equivalent to moe_expert_ffn_verify with T = 1.
 * An expert id outside [0, E) is device data: the call records MOE_ERR_INVALID_ARG in the workspace status word.
 *   y is then untouched for MOE_LAYOUT_TC; for MOE_LAYOUT_DECODE its contents are unspecified. After any device
 *   error, re-zero the workspace with moe_workspace_init() before its next use.
 * Numerics depend on the layer's layout; in both the weights are exact and the sums are fp32.
 *   MOE_LAYOUT_DECODE (mat-vec kernels, every format): x is rescaled per token by a power of two and held in
 *   binary16 (exact for every element within 2^-28 of the token's largest |x|); h is fp32, rescaled per (expert,
 *   token) by a power of two into binary16 for the down projection.
 *   MOE_LAYOUT_TC (MXFP4, block-scaled tcgen05 MMAs, "quantization" glossary, "MXFP4"): x, and h = SiLU(g) * u
 *   formed in fp32, are each carried as the sum of 6 E2M1 parts per 32-block with their own E8M0 exponents
 *   (part p at exponent e0 - 2p quantises what parts 0..p-1 left). The error of an element is below 1/3072 of the
 *   largest |value| of ITS 32-block, not of the element: in a block with one outlier, the other 31 elements carry
 *   errors up to ~outlier/3072. The parity tests hold y to 1e-3 * sum|terms| per element on N(0,1) x, on x with
 *   one element per block scaled by 2^8 .. 2^12 (also over zero weight columns), Student-t(3) x, and x with
 *   exact zeros and bf16 subnormals. A block holding NaN or infinity makes its parts NaN (E8M0 exponent 255). */
moe_status_t moe_expert_ffn_decode(const moe_layer_t* layer, const void* x_bf16, const int32_t* idx, const float* w,
                                   int32_t k, float* y, void* y_bf16, int32_t accumulate, void* ws, size_t ws_bytes,
                                   void* stream);

/* Verify, T tokens (1 <= T <= 8) sharing one sweep of the union of their experts' weights.
 * Row t of y is bit-identical to moe_expert_ffn_decode of token t with the same idx/w rows.
 *   x_bf16 [T, H]; idx [T, k]; w [T, k]; y [T, H]; y_bf16 [T, H] or NULL. */
moe_status_t moe_expert_ffn_verify(const moe_layer_t* layer, const void* x_bf16, int32_t T, const int32_t* idx,
                                   const float* w, int32_t k, float* y, void* y_bf16, int32_t accumulate, void* ws,
                                   size_t ws_bytes, void* stream);

/* Router and expert FFN of T tokens (1 <= T <= 8) in one launch, for a MOE_LAYOUT_TC MXFP4 layer with E <= 256
 * ("Mixed-precision compression of DeepSeek-V4-Flash", "The recipe": F16 router, softmax top-6 of 256 routed
 * experts; the fused always-on neighbours of the expert FFN). The kernel first computes the router logits across
 * the whole grid (workspace scratch), every CTA then selects each token's top-k, and the FFN follows.
 *   router_w_f16 [E, H] fp16 and x_bf16 [T, H] (both 16-byte aligned); idx [T, k] int32 and w [T, k] fp32 are
 *   OUTPUTS, bit-identical to moe_route_topk's for the same router and x; y [T, H] (and y_bf16) are bit-identical
 *   to moe_expert_ffn_verify's with that idx / w. Workspace as for moe_expert_ffn_verify.
 *   Errors: MOE_ERR_UNSUPPORTED_FORMAT (other layout or format), MOE_ERR_SHAPE (T, k, E out of range). */
moe_status_t moe_route_expert_ffn(const moe_layer_t* layer, const void* router_w_f16, const void* x_bf16, int32_t T,
                                  int32_t k, int32_t* idx, float* w, float* y, void* y_bf16, int32_t accumulate,
                                  void* ws, size_t ws_bytes, void* stream);

/* Decode of one token exactly like moe_expert_ffn_decode, but without a workspace argument: its scratch is a
 * fixed array of 2,101,248 bytes inside the library (one per GPU that loads it, kept until the process exits).
 * The pages have no counterpart; it exists for callers that cannot allocate device memory (a plugin given only
 * its input and output buffers, code under a memory budget owned by another allocator).
 *   Layout MOE_LAYOUT_DECODE, any format. Limits: k <= 8 and H, I <= 4096 (MOE_ERR_WORKSPACE_TOO_SMALL /
 *   MOE_ERR_SHAPE otherwise). It calls no allocation routine. The first call on a device looks up the array's
 *   device address (cudaGetSymbolAddress) with that device current and keeps it for the life of the process; make
 *   that first call before any stream capture, and do not call it again on a device after cudaDeviceReset().
 *   Every call shares the array and clears its counters and status word first (an asynchronous memset on
 *   `stream`). Calls that overlap on the GPU (other streams, other threads) race on the array and must be
 *   serialised by the caller. Its results are bit-identical to moe_expert_ffn_decode's with a workspace. */
moe_status_t moe_expert_ffn_decode_static(const moe_layer_t* layer, const void* x_bf16, const int32_t* idx,
                                          const float* w, int32_t k, float* y, void* y_bf16, int32_t accumulate,
                                          void* stream);
/* Device status word (MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_INVALID_ARG for an expert id >= E) left by the most
 * recent moe_expert_ffn_decode_static() on the current device: synchronises `stream`, then reads it. The next
 * static call clears it. No counterpart on the pages. */
moe_status_t moe_static_device_status(void* stream);

/* ---------------------------------------------------------------- speculative acceptance ------------------------ */

/* Acceptance of K drafted tokens after the verify sweep that scored them ("Mixed-precision compression of
 * DeepSeek-V4-Flash" (lumirain.cn), "What compression does not solve": a draft x is kept with probability
 * min(1, p(x) / q(x)); on a rejection the token is drawn from max(p - q, 0), normalised, which keeps the target's
 * distribution exactly).
 *   p [K+1, V] fp32: the target's distribution at each drafted position and after the last draft;
 *   q [K, V] fp32: the drafter's distribution at each drafted position;
 *   draft [K] int32: the drafted tokens; u [K+1] fp32 uniforms in [0, 1): u[k] decides draft k, u[K] drives the
 *   one draw. All are device pointers; the caller owns them.
 *   result [2] int32 (device): result[0] = n, the drafts kept (the first n, in order); result[1] = the token
 *   drawn after them: from the normalised max(p_n - q_n, 0) if draft n was rejected (from p_n if that residual
 *   has no mass), from p_K if all K were kept; -1 if the row has no mass.
 *   Arithmetic: draft k is kept when u[k] < p_k(d) / q_k(d) (one fp32 division: q = 0 < p keeps, p = q = 0
 *   rejects); the draw is an exact integer inverse CDF: weights clamped to [0, 1] (NaN as 0) scaled to
 *   floor(r 2^40), threshold floor(floor(u 2^32) * total / 2^32), the smallest v whose running sum exceeds it.
 *   The same inputs always give the same tokens.
 *   Limits: 0 <= K <= 8, 1 <= V <= 2^22; 4-byte aligned pointers; q and draft may be NULL when K = 0.
 *   A draft id outside [0, V) is device data: the call then writes n = -1 and token -1.
 *   Errors: MOE_ERR_INVALID_ARG (null or misaligned pointer), MOE_ERR_SHAPE (K or V out of range), both before
 *   any launch. One CTA; runs on `stream`. */
moe_status_t moe_spec_accept(const float* p, const float* q, int32_t K, int32_t V, const int32_t* draft,
                             const float* u, int32_t* result, void* stream);

/* ---------------------------------------------------------------- prefill --------------------------------------- */

/* Workspace bytes for moe_expert_grouped_gemm_prefill of up to T_max tokens with top-k (0 for unsupported sizes).
 * Initialise it once with moe_workspace_init(); its first word is the device status word like the decode
 * workspace's, read with moe_get_device_status(). */
size_t moe_prefill_workspace_bytes(const moe_layer_t* layer, int32_t T_max, int32_t k);

/* Prefill of T tokens: y[t] = sum_r w[t,r] * FFN_{idx[t,r]}(x[t]) computed as grouped dense contractions on the
 * tensor cores ("Mixed-precision compression of DeepSeek-V4-Flash", prefill throughput; "quantization" glossary,
 * "GPU compute": block-scaled MXFP4 tensor-core instructions; its "V4.1 Flash" section names the E4M3 sibling
 * format with the same per-32 E8M0 exponent, used here for the activations).
 *   Numerics: x is quantised to MXFP8 per 32 along H (E4M3 codes, e = clamp(k + 127, 1, 254) with k the smallest
 *   integer such that amax <= 448 * 2^k, codes = E4M3 round-to-nearest-even of x * 2^(127 - e)); g and u are
 *   accumulated in fp32; h = SiLU(g) * u in fp32 is quantised the same way per 32 along I; the down projection
 *   accumulates in fp32; y sums the k expert outputs in rank order in fp32.
 *   layer: fmt MXFP4, layout MOE_LAYOUT_TC, 1 <= E <= 1024. x_bf16 [T, H] bf16 (16-byte aligned);
 *   idx [T, k] int32; w [T, k] fp32; 1 <= k <= 8. y [T, H] fp32 (16-byte aligned) and/or y_bf16 [T, H] bf16
 *   (8-byte aligned; round-to-nearest-even copy of y); either may be NULL, not both.
 *   ws: moe_prefill_workspace_bytes(layer, T_max >= T, k) bytes, 256-byte aligned.
 *   An expert id outside [0, E) sets the device status MOE_ERR_INVALID_ARG and that (token, rank) pair
 *   contributes nothing. Consecutive calls on one stream may share a workspace; calls that overlap on the GPU
 *   must not. */
moe_status_t moe_expert_grouped_gemm_prefill(const moe_layer_t* layer, const void* x_bf16, int32_t T,
                                             const int32_t* idx, const float* w, int32_t k, float* y, void* y_bf16,
                                             void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- between layers --------------------------------- */

/* RMS normalisation of a layer's output into the next layer's bf16 input, for stacks of layers (the model of
 * "Mixed-precision compression of DeepSeek-V4-Flash", "The recipe", normalises the hidden state before each MoE
 * layer; a stack that passed y on unnormalised would drift to zero or overflow):
 *   x_bf16[t, i] = bf16_rne( y[t, i] * r ), r = fp32( 1 / sqrt(mean_i y[t, i]^2 + eps) ), no learned gain;
 *   the sum of squares (fixed order per token) and r in fp64, the product in fp32.
 *   y [T, H] fp32 (4-byte aligned), x_bf16 [T, H] bf16 (2-byte aligned); 1 <= H <= 2^20, T >= 1, eps >= 0.
 *   A token's result does not depend on the other tokens. NaN and infinity propagate.
 *   Errors: MOE_ERR_INVALID_ARG (null or misaligned pointer), MOE_ERR_SHAPE, before any launch. */
moe_status_t moe_rms_norm_bf16(const float* y, int32_t T, int32_t H, float eps, void* x_bf16, void* stream);

/* ---------------------------------------------------------------- debug (tests only) ----------------------------- */

/* Unpack expert `expert` of a packed matrix back to fp32 values [rows, K] (rows = I for each of gate and up,
 * written as [2, I, H]; rows = H for down, [H, I]). For bit-exact checks of the layout. */
moe_status_t moe_debug_unpack(moe_format_t fmt, moe_layout_t layout, moe_matrix_t kind, const void* packed,
                              int64_t H, int64_t I, int64_t expert, float* out, void* stream);

/* Runs a one-CTA kernel that waits on a flag nothing sets, with a limit of `limit_us` microseconds, then records
 * MOE_ERR_DEVICE_TIMEOUT in the workspace status word and returns. Tests the bounded-wait path. */
moe_status_t moe_debug_timeout_probe(void* ws, size_t ws_bytes, int32_t limit_us, void* stream);

/* moe_expert_grouped_gemm_prefill with test hooks: if gu_dump is not NULL, the gate/up GEMM also writes its fp32
 * accumulators g and u to gu_dump [rows_max][2I] (row = the pair's row in the sorted buffers, g then u); if
 * offsets is not NULL it receives 8 values describing the workspace: rows_max, tiles_max, and the byte offsets of
 * n_tiles (uint32), tile_first (int32 [tiles]: compact index of each tile's first pair), pair_row (int32 [T*k]:
 * row of pair (t, r), -1 for an invalid id), xq, hq (the sorted MXFP8 x and h: for each 128-row tile and
 * 128-column group, 16384 bytes of E4M3 codes [128 rows][128] then the 512-byte exponent block permuted as in
 * MOE_LAYOUT_TC) and dout (fp32 [T*k][H], compact pair order: tile_first[row / 128] + row % 128). */
moe_status_t moe_debug_prefill(const moe_layer_t* layer, const void* x_bf16, int32_t T, const int32_t* idx,
                               const float* w, int32_t k, float* y, void* y_bf16, void* ws, size_t ws_bytes,
                               float* gu_dump, int64_t* offsets, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BIT_MOE_DECODE_GB300_MOE_H */
