/*
 * vg_fused.h -- C ABI of libvg_fused.so: fused residual-add + RMSNorm -> FP8
 * and SiLU-and-mul -> FP8 quantisation on one GB300 (sm_103a).
 *
 * Operations (cited by page title and section):
 *   "Fusion torch.compile passes" (data-sketchers.com wiki, vLLM
 *   design-fusions page), section "RMSNorm + Quantization (fuse_norm_quant)":
 *   rms_norm(x) -> quant_fp8(y) and fused_add_rms_norm(x, residual) ->
 *   quant_fp8(y) in one kernel, the residual updated in place, with FP8
 *   static per-tensor, dynamic per-token and dynamic per-token-group (128/64)
 *   scales.  Section "SiLU+Mul + Quantization (fuse_act_quant)":
 *   silu_and_mul of the gate-up projection -> quant_fp8 in one kernel,
 *   without materialising the post-activation tensor.  "Quick Reference"
 *   table: both fusions apply for every num_tokens.  Section "MLA Dual
 *   RMSNorm (fuse_mla_dual_rms_norm)": the paired q_c / kv_c RMSNorms of MLA
 *   attention in one kernel, and its per-token-quant variant (q to FP8 with
 *   a per-token scale, kv in bf16).  Section "RMSNorm + Padding
 *   (fuse_act_padding)": residual add + RMSNorm written into a padded bf16
 *   row.  Section "QK Norm + RoPE (enable_qk_norm_rope_fusion)": per-head
 *   RMSNorm of Q and K, then the rotary embedding, in place on qkv.  The
 *   "Quick Reference" table also names FP4 outputs of both fusions and the
 *   "Support Matrix" NVFP4 and DeepGEMM-style per-group FP8 on sm100: the
 *   NVFP4 entry points and the per-group scale options (UE8M0,
 *   column-major) below.
 *
 * Numerics (the pages give no formulas; these are the readings the library
 * implements):
 *   r   = bf16(x + residual)                       (fp32 add, RNE to bf16)
 *   y   = r / sqrt(mean(r^2) + eps) * weight       (fp32, never rounded to bf16)
 *   a   = gate / (1 + exp(-gate)) * up             (fp32, never rounded to bf16)
 *   q   = e4m3(y / s)    RNE, saturating to +-448, OCP E4M3FN encoding
 *   s   = static: the given fp32 scale
 *         per-token: fp32(max(amax over the row, 1e-10f) / 448)
 *         per-group: fp32(max(amax over G columns, 1e-10f) / 448)
 *   The kernels multiply by 1/s, computed once per row or group.
 *   A norm with a bf16 output (the MLA dual norm, the padded norm) rounds y
 *   once, to nearest even bf16, as the exact value would round (the QK
 *   norm + RoPE: see its entry point).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing, keeps no per-call state, never
 *     synchronises, and launches only on `stream` (NULL = legacy default
 *     stream).  Calls are asynchronous and may be captured in a CUDA graph.
 *   - Stream order: every output is visible to whatever runs after the call
 *     in stream order.  Every kernel is launched with programmatic
 *     dependent launch: it may start while the previous kernel in the
 *     stream is still draining, waits for it (griddepcontrol.wait) before
 *     it reads or writes any memory -- it only asks its first input rows
 *     into L2 before the wait, which cannot return stale data, since L2
 *     also takes every write of the previous kernel -- and signals
 *     griddepcontrol.launch_dependents once its loads are issued, before
 *     q, scale and residual_out are written.  A consumer launched
 *     after it with programmatic dependent launch too must therefore wait
 *     on the grid dependency (cudaGridDependencySynchronize() or
 *     griddepcontrol.wait) before it reads these outputs; an ordinary
 *     launch, a copy or an event needs nothing extra.
 *   - bf16 tensors are passed as uint16_t bit patterns, fp8 outputs as
 *     uint8_t E4M3 codes.  All tensors are dense and row-major, except the
 *     MLA dual norm's two inputs, which are read through a row stride.
 *   - Every argument is validated on the host before any launch; a
 *     validation error returns its status and launches nothing.  A launch
 *     failure returns VG_ERR_CUDA.  num_tokens == 0 returns VG_OK without
 *     launching.
 *   - Alignment: every bf16 / fp8 tensor pointer must be 16-byte aligned,
 *     `scale` 4-byte aligned.  The row length (hidden or inter) must be a
 *     multiple of 8 and at most VG_MAX_ROW.
 *   - Aliasing: residual_out may equal residual exactly (in-place update).
 *     Any other overlap between an output and any other tensor is undefined.
 *   - Device: compute capability 10.3 (GB300) only; other devices return
 *     VG_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef VG_FUSED_H
#define VG_FUSED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t from cuda_runtime.h. */
struct CUstream_st;
typedef struct CUstream_st *vg_stream_t;

#define VG_ABI_VERSION 3
#define VG_MAX_ROW 32768 /* largest hidden / inter a row-resident kernel holds */

typedef enum {
    VG_SCALE_STATIC = 0,    /* s given: scale[0], fp32, read on the device         */
    VG_SCALE_PER_TOKEN = 1, /* s computed per row: scale[T] written                 */
    VG_SCALE_PER_GROUP = 2  /* s per G columns: scale[T, n/G] written, row-major    */
} vg_scale_mode;

/*
 * Per-group options, or-ed into `mode` with VG_SCALE_PER_GROUP only (any
 * other use is VG_ERR_BAD_MODE): the scale formats a GEMM on sm100 consumes
 * (the pages' "Support Matrix" pairs per-group FP8 there with DeepGEMM;
 * E8M0 is from the OCP Microscaling spec).
 *   VG_SCALE_UE8M0         each scale is the smallest power of two
 *                          >= max(amax, 1e-10f) / 448 (stored as fp32);
 *                          codes are e4m3(y / s)
 *   VG_SCALE_COLUMN_MAJOR  scale (t, g) is stored at [g, t] of an fp32
 *                          [n/G, T4] tensor, T4 = T rounded up to a multiple
 *                          of 4 (16-byte rows); columns [T, T4) are not written
 */
#define VG_SCALE_UE8M0 0x100
#define VG_SCALE_COLUMN_MAJOR 0x200

typedef enum {
    VG_OK = 0,
    VG_ERR_NULL_PTR = 1,           /* a required pointer is NULL, or residual_out
                                      and residual are not both set or both NULL  */
    VG_ERR_BAD_SHAPE = 2,          /* num_tokens < 0, row length not a multiple
                                      of 8, < 8, or > VG_MAX_ROW                  */
    VG_ERR_MISALIGNED = 3,         /* a tensor pointer breaks the alignment rule */
    VG_ERR_BAD_MODE = 4,           /* mode is not a vg_scale_mode (with valid
                                      per-group options)                          */
    VG_ERR_BAD_GROUP = 5,          /* per-group with group_size not 64 or 128, or
                                      not dividing the row length                 */
    VG_ERR_UNSUPPORTED_DEVICE = 6, /* current device is not compute capability 10.3 */
    VG_ERR_CUDA = 7                /* a CUDA runtime call or launch failed        */
} vg_status;

/*
 * Residual add + RMSNorm -> FP8 ("RMSNorm + Quantization (fuse_norm_quant)").
 *
 *   q            out  uint8  [T, H]  E4M3 codes of y / s
 *   residual_out out  uint16 [T, H]  bf16 r = bf16(x + residual); may equal
 *                                    `residual` (in place).  NULL iff residual
 *                                    is NULL.
 *   scale        STATIC: in fp32 [1]; PER_TOKEN: out fp32 [T];
 *                PER_GROUP: out fp32 [T, H / group_size]
 *   x            in   uint16 [T, H]  bf16
 *   residual     in   uint16 [T, H]  bf16, or NULL for the plain
 *                                    rms_norm(x) -> quant_fp8 variant (r = x)
 *   weight       in   uint16 [H]     bf16
 *   num_tokens T >= 0; hidden H: multiple of 8, 8 <= H <= VG_MAX_ROW
 *   eps          added to mean(r^2) inside the square root
 *   mode         vg_scale_mode, with VG_SCALE_PER_GROUP optionally or-ed
 *                with VG_SCALE_UE8M0 / VG_SCALE_COLUMN_MAJOR; group_size 64
 *                or 128 (PER_GROUP only, ignored otherwise)
 */
vg_status vg_fused_add_rms_norm_fp8(uint8_t *q, uint16_t *residual_out, float *scale,
                                    const uint16_t *x, const uint16_t *residual,
                                    const uint16_t *weight, int64_t num_tokens,
                                    int64_t hidden, float eps, int32_t mode,
                                    int32_t group_size, vg_stream_t stream);

/*
 * SiLU(gate) * up -> FP8 ("SiLU+Mul + Quantization (fuse_act_quant)").
 *
 *   q        out uint8  [T, I]  E4M3 codes of a / s
 *   scale    STATIC: in fp32 [1]; PER_TOKEN: out fp32 [T];
 *            PER_GROUP: out fp32 [T, I / group_size]
 *   gate_up  in  uint16 [T, 2I] bf16: gate = columns [0, I), up = [I, 2I)
 *   num_tokens T >= 0; inter I: multiple of 8, 8 <= I <= VG_MAX_ROW
 *   mode, group_size as above.  SiLU has no epsilon, so there is none here.
 */
vg_status vg_silu_mul_fp8(uint8_t *q, float *scale, const uint16_t *gate_up,
                          int64_t num_tokens, int64_t inter, int32_t mode,
                          int32_t group_size, vg_stream_t stream);

/*
 * NVFP4 outputs of both fusions.  The "Quick Reference" table names FP4 as an
 * output of "RMSNorm + Quantization" and of "SiLU+Mul + Quantization" and the
 * "Support Matrix" lists NVFP4 dynamic quantisation on sm100 and later; the
 * pages define neither, so the library takes NVIDIA's public NVFP4 format:
 *   elements  E2M1 (OCP Microscaling FP4: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}),
 *             RNE, saturating at 6; two a byte, column 2i in the low nibble
 *   blocks    16 consecutive columns of a row, one E4M3 code each:
 *             sf = e4m3(gs * amax / 6), amax over the block's y (or a)
 *   elements  q = e2m1(y * gs / decode(sf)); a block with sf == 0 gives +0
 *   gs        the fp32 per-tensor scale, read from device memory
 * The block code is the one the exact gs * amax / 6 rounds to.  Element codes
 * differ from the exact value's only where it lies within ~2^-19 (relative)
 * of an E2M1 midpoint, by one code.
 *
 *   q4            out uint8 [T, H/2] (or [T, I/2])  packed E2M1 codes
 *   block_scale   out uint8 [T, H/16] (or [T, I/16]) E4M3 codes, row-major
 *   global_scale  in  fp32 [1], device, > 0 and finite
 *   the other arguments as for vg_fused_add_rms_norm_fp8 / vg_silu_mul_fp8;
 *   the row length must be a multiple of 16 (else VG_ERR_BAD_SHAPE).
 *   block_scale has no alignment rule; global_scale must be 4-byte aligned.
 */
vg_status vg_fused_add_rms_norm_nvfp4(uint8_t *q4, uint8_t *block_scale, uint16_t *residual_out,
                                      const uint16_t *x, const uint16_t *residual,
                                      const uint16_t *weight, const float *global_scale,
                                      int64_t num_tokens, int64_t hidden, float eps,
                                      vg_stream_t stream);
vg_status vg_silu_mul_nvfp4(uint8_t *q4, uint8_t *block_scale, const uint16_t *gate_up,
                            const float *global_scale, int64_t num_tokens, int64_t inter,
                            vg_stream_t stream);

/*
 * Residual add + RMSNorm into a padded bf16 row ("RMSNorm + Padding
 * (fuse_act_padding)"): the normalised row stays bf16 and is written into a
 * row of padded_hidden columns whose tail is zero, the width the next GEMM
 * needs.
 *
 *   out          out  uint16 [T, padded_hidden]  bf16: columns [0, H) are
 *                                    bf16(y) (one rounding), [H, padded) zero
 *   residual_out out  uint16 [T, H]  as for vg_fused_add_rms_norm_fp8 (may
 *                                    equal `residual`; NULL iff residual is)
 *   x, residual, weight, num_tokens, hidden, eps  as for
 *                                    vg_fused_add_rms_norm_fp8
 *   padded_hidden  >= hidden, a multiple of 8, at most 2 * VG_MAX_ROW
 *                  (else VG_ERR_BAD_SHAPE)
 * `out` must not overlap any other tensor.
 */
vg_status vg_fused_add_rms_norm_pad(uint16_t *out, uint16_t *residual_out, const uint16_t *x,
                                    const uint16_t *residual, const uint16_t *weight,
                                    int64_t num_tokens, int64_t hidden, int64_t padded_hidden,
                                    float eps, vg_stream_t stream);

/*
 * MLA dual RMSNorm ("MLA Dual RMSNorm (fuse_mla_dual_rms_norm)"): in one
 * launch,
 *   q_out  = bf16(rms_norm(q_c,  q_weight,  eps_q))
 *   kv_out = bf16(rms_norm(kv_c, kv_weight, eps_kv))
 * with rms_norm(x, w, eps)_j = x_j / sqrt(mean(x^2) + eps) * w_j.
 *
 *   q_out      out uint16 [T, q_dim]   bf16, dense
 *   kv_out     out uint16 [T, kv_dim]  bf16, dense
 *   q_c        in  uint16 bf16; row t is q_c[t * q_stride + j], j < q_dim
 *   q_stride   elements between rows of q_c: >= q_dim, a multiple of 8
 *              (q_c and kv_c are usually column slices of one projected
 *              [T, q_dim + kv_dim + rope] tensor, both with its row length)
 *   q_weight   in  uint16 [q_dim] bf16
 *   kv_c, kv_stride, kv_weight   the same for the kv side
 *   num_tokens T >= 0; q_dim, kv_dim: multiples of 8 in [8, VG_MAX_ROW]
 *   eps_q, eps_kv  each side's epsilon
 * Outputs must not overlap any input or each other.  A stride < dim or not
 * a multiple of 8 is VG_ERR_BAD_SHAPE.
 */
vg_status vg_fused_mla_dual_rms_norm(uint16_t *q_out, uint16_t *kv_out, const uint16_t *q_c,
                                     int64_t q_stride, const uint16_t *q_weight,
                                     const uint16_t *kv_c, int64_t kv_stride,
                                     const uint16_t *kv_weight, int64_t num_tokens,
                                     int64_t q_dim, int64_t kv_dim, float eps_q,
                                     float eps_kv, vg_stream_t stream);

/*
 * The per-token-quant variant ("MLA Dual RMSNorm", FP8 attention with a
 * per-token q_b_proj): q goes through rms_norm -> dynamic per-token FP8 as
 * in vg_fused_add_rms_norm_fp8 without a residual, kv stays bf16.
 *
 *   q_fp8    out uint8 [T, q_dim]  E4M3 codes of y / s
 *   q_scale  out fp32  [T]         s = fp32(max(amax of the q row, 1e-10f) / 448)
 *   kv_out   out uint16 [T, kv_dim] bf16
 *   the inputs and sizes as for vg_fused_mla_dual_rms_norm.
 */
vg_status vg_fused_mla_dual_rms_norm_per_token_quant(
    uint8_t *q_fp8, float *q_scale, uint16_t *kv_out, const uint16_t *q_c, int64_t q_stride,
    const uint16_t *q_weight, const uint16_t *kv_c, int64_t kv_stride, const uint16_t *kv_weight,
    int64_t num_tokens, int64_t q_dim, int64_t kv_dim, float eps_q, float eps_kv,
    vg_stream_t stream);

/*
 * Per-head QK RMSNorm + rotary embedding, in place ("QK Norm + RoPE
 * (enable_qk_norm_rope_fusion)").  For every token t and every Q head
 * (weight q_weight) and K head (weight k_weight):
 *   y_j = x_j / sqrt(mean(x^2) + eps) * w_j                 over the head's D columns
 *   o_a = y_a c_i - y_b s_i,  o_b = y_b c_i + y_a s_i       i < D/2
 * with c_i = cos_sin_cache[pos_t, i], s_i = cos_sin_cache[pos_t, D/2 + i]
 * and the pairs (a, b) = (i, i + D/2) when is_neox, else (2i, 2i + 1); the
 * head is overwritten with bf16(o), rounded once from an fp32 value within
 * ~2^-20 (relative) of the exact o: so each output is the correctly rounded
 * bf16, or one ulp from it where the exact o lies within ~2^-20 of a bf16
 * rounding midpoint.  V heads are not touched.
 *
 *   qkv            in/out uint16 [T, (Hq + 2 Hkv) * D] bf16: Q heads, then K
 *                  heads, then V heads, D contiguous columns each
 *   q_weight, k_weight  in uint16 [D] bf16 (NULL allowed for zero heads)
 *   cos_sin_cache  in fp32 [max_position, D]: cos in columns [0, D/2), sin
 *                  in [D/2, D)
 *   positions      in int64 [T] (8-byte aligned).  A position outside
 *                  [0, max_position) leaves that token's heads unchanged and
 *                  sets VG_DEVICE_BAD_POSITION (vg_device_status).
 *   num_q_heads Hq >= 0, num_kv_heads Hkv >= 0, Hq + Hkv >= 1,
 *   Hq + 2 Hkv <= 4096; head_dim D in {64, 128, 256}; max_position >= 1
 */
vg_status vg_fused_qk_norm_rope(uint16_t *qkv, const uint16_t *q_weight, const uint16_t *k_weight,
                                const float *cos_sin_cache, const int64_t *positions,
                                int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int64_t max_position, float eps, int32_t is_neox,
                                vg_stream_t stream);

/*
 * Device-side status of the library's kernels on the current device (no
 * counterpart on the pages; the pipelined kernels' own failure report).
 * Every wait in the library's kernels is bounded; a wait that gives up sets
 * VG_DEVICE_WAIT_TIMEOUT here, waits (bounded) for its own copies and
 * returns, so the context stays usable and the outputs of that call are
 * not valid.  Writes the flags seen since the last reset to *flags and,
 * if reset != 0, clears them.  Synchronous (it reads device memory); not
 * for use inside stream capture.  Returns VG_ERR_NULL_PTR, VG_ERR_CUDA or
 * VG_OK.
 */
#define VG_DEVICE_WAIT_TIMEOUT 1u
#define VG_DEVICE_BAD_POSITION 2u /* vg_fused_qk_norm_rope: a position out of range */
/* Debug builds only (compiled with VG_DEBUG_CHECKS, a test copy of the
 * library): a kernel computed a store or copy address outside the tensor it
 * belongs to; the access was skipped. */
#define VG_DEVICE_OUT_OF_BOUNDS 4u
vg_status vg_device_status(uint32_t *flags, int32_t reset);

/* Static English text for a status code (never NULL). */
const char *vg_status_string(vg_status status);

/* VG_ABI_VERSION of the library that is loaded. */
int32_t vg_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VG_FUSED_H */
