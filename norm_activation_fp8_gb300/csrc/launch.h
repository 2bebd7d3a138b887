// launch.h -- internal (non-ABI) declarations shared by the library's .cu files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vg {

// kStatic / kPerToken / kPerGroup are vg_scale_mode; kBf16Pad is the
// norm's bf16 output into a padded row (no quantisation); kPerGroupX is
// per-group with scale options (UE8M0 scales and/or the column-major
// layout), kept apart so that plain per-group code stays as it is.
enum ScaleMode : int { kStatic = 0, kPerToken = 1, kPerGroup = 2, kBf16Pad = 3, kPerGroupX = 4,
                       kNvfp4 = 5 /* E2M1 codes, E4M3 scales per 16 columns */ };

// How a row-wise kernel covers a [T, n] tensor: each row is split into
// nch = n/8 chunks of 16 bytes; `ntr` threads (a multiple of 32) own a row,
// thread i holding chunks i, i + ntr, ..., i + (vpt-1)*ntr; a CTA carries
// `rpc` rows, so it has ntr * rpc threads.
struct RowPlan {
  int vpt;
  int ntr;
  int rpc;
  int64_t grid;
  int segs = 1;  // column segments per row (row-state-free SiLU modes only)
  bool dense = false;  // SiLU per-group: the four-CTAs-per-SM instance
  int block() const { return ntr * rpc; }
};

// Picks the plan for nch chunks per row (nch <= 4096) on a device with `sms`
// SMs: with few rows (T < 2 sms) one row per CTA and as few chunks per
// thread as fit 512 threads; otherwise at least `min_vpt` chunks per thread
// (more if a row would need more than 512 threads), short rows packed
// several to a CTA.
RowPlan plan_rows(int64_t T, int nch, int min_vpt, int sms);
RowPlan plan_silu(int64_t T, int nch, int mode, int sms);

struct NormArgs {
  uint8_t *q;
  uint16_t *res_out;
  float *scale;
  const uint16_t *x;
  const uint16_t *res;
  const uint16_t *w;
  int64_t T;
  int32_t H;
  int32_t nch;     // H / 8
  int32_t ntr;     // threads per row
  int32_t rpc;     // rows per CTA
  int32_t gch;     // chunks per scale group (G / 8), per-group mode only
  int32_t ngroups; // H / G, per-group mode only
  float eps;
  float inv_h;     // 1 / H
  uint16_t *out16; // kBf16Pad: bf16 output rows of nch_pad chunks
  int32_t nch_pad; // kBf16Pad: padded row length / 8
  // per-group scale (t, g) lives at scale[t * s_ts + g * s_gs] (row-major:
  // s_ts = ngroups, s_gs = 1; column-major: s_ts = 1, s_gs = T rounded up
  // to 4); ue8m0: power-of-two scales
  int32_t s_ts;
  int32_t s_gs;
  int32_t ue8m0;
  uint8_t *sf8;    // kNvfp4: E4M3 block scale codes [T, H/16]; q holds [T, H/2]
  int32_t pf_ctas; // CTAs below this index prefetch their first rows into L2
  int32_t fastq;   // dynamic FP8 codes in the two-multiply form where allowed
};

struct SiluArgs {
  uint8_t *q;
  float *scale;
  const uint16_t *gate_up;
  int64_t T;
  int32_t I;
  int32_t nch;
  int32_t ntr;
  int32_t rpc;
  int32_t gch;
  int32_t ngroups;
  int32_t s_ts;    // per-group scale (t, g) at scale[t * s_ts + g * s_gs]
  int32_t s_gs;
  int32_t ue8m0;   // power-of-two per-group scales
  uint8_t *sf8;    // kNvfp4: E4M3 block scale codes [T, I/16]; q holds [T, I/2]
  int32_t pf_ctas; // CTAs below this index prefetch their first rows into L2
};

cudaError_t launch_norm_fp8(NormArgs a, int mode, const RowPlan &plan, cudaStream_t stream);

// Persistent TMA-pipelined norm kernel: `grid` CTAs of `block` threads (one
// row at a time, vpt chunks per thread), `stages` rows staged ahead.
struct TmaPlan {
  int vpt;
  int block;
  int stages;
  int64_t grid;
  size_t smem;  // dynamic shared memory to request (>= the layout's need)
};
constexpr size_t kTmaMaxSmem = 227 * 1024;  // opt-in limit per CTA (static + dynamic)

// Lets `kern` use dynamic shared memory up to the opt-in limit minus its own
// static shared memory (asking for more fails the call).
inline cudaError_t opt_in_dynamic_smem(const void *kern) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(kTmaMaxSmem - fa.sharedSizeBytes));
}
size_t norm_tma_smem_bytes(int H, bool res, int stages, int block, int vpt, int slots);
cudaError_t launch_norm_fp8_tma(NormArgs a, int mode, const TmaPlan &plan, cudaStream_t stream);

// Reads (and optionally clears) the norm kernels' device status word;
// synchronous.  0xFFFFFFFF if it could not be read.
uint32_t read_norm_status(bool reset);
cudaError_t launch_silu_fp8(SiluArgs a, int mode, const RowPlan &plan, cudaStream_t stream);


// Persistent TMA-staged per-token SiLU kernel: `grid` CTAs of `block`
// threads (vpt chunks each), one row at a time in `nseg` staged segments.
struct SiluTmaPlan {
  int vpt;
  int block;
  int nseg;  // column segments of a row, one stage each (1 or 2)
  int64_t grid;
  size_t smem;  // dynamic shared memory to request (>= the stages' need)
};
size_t silu_tma_token_smem_bytes(int I, int nseg);
cudaError_t launch_silu_fp8_tma_token(SiluArgs a, const SiluTmaPlan &plan, cudaStream_t stream);
uint32_t read_silu_status(bool reset);

// MLA dual RMSNorm: side 0 is the q row, side 1 the kv row of each token.
struct MlaArgs {
  const uint16_t *src[2];  // q_c, kv_c (strided rows)
  const uint16_t *w[2];
  int64_t stride[2];       // elements between rows of src
  uint16_t *out[2];        // bf16 outputs (out[0] unused when q goes to fp8)
  uint8_t *q8;             // fp8 q output (per-token-quant variant)
  float *q_scale;          // [T]
  int64_t T;
  int32_t nch[2];          // chunks per row
  int32_t thr[2];          // threads per row (multiples of 32)
  int32_t rpc;             // tokens per CTA
  float eps[2];
  float n[2];              // row lengths
  float inv_n[2];          // 1 / row length
  int32_t pf_ctas;         // CTAs below this index prefetch their rows into L2
};

// vpt == 0: the warp-per-token kernel (block/32 tokens per CTA);
// otherwise the warp-group kernel (rpc tokens per CTA).
struct MlaPlan {
  bool spread = false;  // warp kernel: tokens dealt out across one wave of CTAs
  int vpt;
  int thr[2];
  int rpc;
  int block;
  int64_t grid;
};
MlaPlan plan_mla(int64_t T, int nq, int nkv, bool q_fp8, int sms);
cudaError_t launch_mla_dual_norm(MlaArgs a, bool q_fp8, const MlaPlan &p, cudaStream_t s);
uint32_t read_mla_status(bool reset);

// QK norm + RoPE, in place on qkv [T, row] with row = (hq + 2 hkv) * D.
struct QkArgs {
  uint16_t *qkv;
  const uint16_t *qw;
  const uint16_t *kw;
  const float *cache;    // [max_pos, D]: cos | sin
  const int64_t *pos;    // [T]
  int64_t T;
  int64_t row;           // elements per token row
  int64_t max_pos;
  int32_t nh;            // heads normalised: hq + hkv
  int32_t hq;
  float eps;
  int32_t pf_ctas;       // tokens below this index prefetch their heads into L2
};
// Device status bit of the rope kernel: a position outside [0, max_pos).
constexpr uint32_t kErrBadPosition = 2u;
cudaError_t launch_qk_norm_rope(const QkArgs &a, int head_dim, bool neox, cudaStream_t s);
uint32_t read_rope_status(bool reset);

}  // namespace vg
