// vg_fused.cu -- the C ABI declared in include/vg_fused.h.
//
// Host side only: validates every argument before launching anything,
// checks the device once per device, picks a row plan from the shape and
// launches on the caller's stream.  No allocation, no synchronisation, no
// per-call state, so every call can be captured in a CUDA graph.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "launch.h"
#include "vg_fused.h"

namespace vg {
namespace {

constexpr int kMaxDevices = 64;
// 0 = not checked yet, 1 = supported (cc 10.3), 2 = unsupported.
std::atomic<int> g_device_state[kMaxDevices];
std::atomic<int> g_device_sms[kMaxDevices];
std::atomic<int> g_device_smem[kMaxDevices];      // shared memory per SM
std::atomic<int> g_device_smem_rsv[kMaxDevices];  // reserved by the system per CTA

// Checks (once per device) that the current device is a GB300 and returns
// its SM count in *sms.
vg_status check_device(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VG_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return VG_ERR_UNSUPPORTED_DEVICE;
  int st = g_device_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, n = 0, smem = 0, rsv = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
      return VG_ERR_CUDA;
    g_device_sms[dev].store(n, std::memory_order_relaxed);
    g_device_smem[dev].store(smem, std::memory_order_relaxed);
    g_device_smem_rsv[dev].store(rsv, std::memory_order_relaxed);
    st = (major == 10 && minor == 3) ? 1 : 2;
    g_device_state[dev].store(st, std::memory_order_release);
  }
  *sms = g_device_sms[dev].load(std::memory_order_relaxed);
  return st == 1 ? VG_OK : VG_ERR_UNSUPPORTED_DEVICE;
}

// Dynamic shared memory for a persistent kernel that must keep exactly
// `ctas` CTAs on an SM: at least `need`, and enough that ctas + 1 of them do
// not fit.  The persistent kernels are launched with programmatic dependent
// launch; without the cap, CTAs of the next launch would take a spare slot
// beside the running ones as soon as it is scheduled, and the later CTAs
// would then pile onto the SMs that free up first, so that some SMs hold
// more CTAs (and rows) than others.  With it, each next CTA takes the slot
// of one that has finished.  Returns `need` if the cap does not fit.
size_t cap_residency_smem(int ctas, size_t need) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return need;
  const size_t per_sm = (size_t)g_device_smem[dev].load(std::memory_order_relaxed);
  const size_t rsv = (size_t)g_device_smem_rsv[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) return need;
  const size_t cap = per_sm / (size_t)(ctas + 1) + 128 - rsv;  // ctas + 1 exceed the SM
  const size_t want = need > cap ? need : (cap + 127) / 128 * 128;
  if (want > kTmaMaxSmem || (size_t)ctas * (want + rsv) > per_sm) return need;
  return want;
}

// Each launch reports its own error through cudaGetLastError(); clear any
// earlier, non-sticky error of this library's runtime first so it is not
// blamed on this call (a sticky, context-level error comes back anyway).
inline void clear_stale_error() { (void)cudaGetLastError(); }

inline bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

vg_status check_row(int64_t num_tokens, int64_t n, int32_t mode_flags, int32_t group_size) {
  const int32_t mode = mode_flags & 0xFF, flags = mode_flags & ~0xFF;
  if (mode != VG_SCALE_STATIC && mode != VG_SCALE_PER_TOKEN && mode != VG_SCALE_PER_GROUP)
    return VG_ERR_BAD_MODE;
  if ((flags & ~(VG_SCALE_UE8M0 | VG_SCALE_COLUMN_MAJOR)) != 0 ||
      (flags != 0 && mode != VG_SCALE_PER_GROUP))
    return VG_ERR_BAD_MODE;
  if ((flags & VG_SCALE_COLUMN_MAJOR) && num_tokens > INT32_MAX - 3)  // T4 must fit int32
    return VG_ERR_BAD_SHAPE;
  if (num_tokens < 0 || num_tokens > INT32_MAX || n < 8 || n % 8 != 0 || n > VG_MAX_ROW)
    return VG_ERR_BAD_SHAPE;
  if (mode == VG_SCALE_PER_GROUP && ((group_size != 64 && group_size != 128) || n % group_size != 0))
    return VG_ERR_BAD_GROUP;
  return VG_OK;
}

// Where scale (t, g) goes and whether it is a power of two, from the mode's
// per-group options.
template <class Args>
void set_scale_layout(Args &a, int32_t mode_flags, int64_t T) {
  const bool col = (mode_flags & VG_SCALE_COLUMN_MAJOR) != 0;
  a.s_ts = col ? 1 : a.ngroups;
  a.s_gs = col ? (int32_t)((T + 3) / 4 * 4) : 1;
  a.ue8m0 = (mode_flags & VG_SCALE_UE8M0) != 0;
}

}  // namespace

RowPlan plan_rows(int64_t T, int nch, int min_vpt, int sms) {
  RowPlan p;
  if (T < 2LL * sms) {
    // Few rows: latency-bound, so spread them -- one row per CTA and the
    // fewest chunks per thread that keep a row within 512 threads.
    p.vpt = 1;
    while (p.vpt < 8 && (nch + p.vpt - 1) / p.vpt > 512) p.vpt *= 2;
    p.ntr = ((nch + p.vpt - 1) / p.vpt + 31) / 32 * 32;
    p.rpc = 1;
  } else if (nch <= 128) {  // one warp per row, eight rows per CTA
    p.ntr = 32;
    p.vpt = nch <= 32 ? 1 : (nch <= 64 ? 2 : 4);
    p.rpc = 8;
  } else {
    p.vpt = min_vpt;
    while (p.vpt < 8 && (nch + p.vpt - 1) / p.vpt > 512) p.vpt *= 2;
    const int per = (nch + p.vpt - 1) / p.vpt;
    p.ntr = (per + 31) / 32 * 32;
    p.rpc = p.ntr <= 128 ? 2 : 1;
  }
  p.grid = (T + p.rpc - 1) / p.rpc;
  return p;
}

// SiLU.  Static / per-group keep no row state: a row is cut into column
// segments of at most 448 threads x VPT chunks (two chunks a thread; static
// four below two rows per SM), each an independent CTA; from two rows per
// SM these run the dense instance (four CTAs per SM).  Rows of <= 64 chunks
// go one warp per row, eight rows per CTA.  Per-token needs the row in one
// CTA: four chunks a thread, up to 1024 threads (fewer chunks when that
// still fits 448 threads).
RowPlan plan_silu(int64_t T, int nch, int mode, int sms) {
  RowPlan p;
  p.rpc = 1;
  p.segs = 1;
  if (mode == VG_SCALE_PER_TOKEN) {
    p.vpt = 4;
    while (p.vpt > 1 && (nch + p.vpt / 2 - 1) / (p.vpt / 2) <= 448) p.vpt /= 2;
  } else if (nch <= 64) {
    p.ntr = 32;
    p.vpt = nch <= 32 ? 1 : 2;
    p.rpc = 8;
    p.grid = (T + p.rpc - 1) / p.rpc;
    return p;
  } else {
    p.dense = T >= 2LL * sms;
    p.vpt = (mode == VG_SCALE_STATIC && !p.dense) ? 4 : 2;
    p.segs = (nch + 448 * p.vpt - 1) / (448 * p.vpt);
  }
  const int per = (nch + p.segs * p.vpt - 1) / (p.segs * p.vpt);
  p.ntr = (per + 31) / 32 * 32;
  p.grid = T;
  return p;
}

// Per-token SiLU from two rows per SM streams through the persistent TMA
// kernel (measured on GB300: from T ~ 300 at I = 14336 and T ~ 256 at
// I = 28672 it beats the register kernel, by up to 18 % at I = 28672; below
// that the register kernel's shorter chain wins).  A row of at least 1024
// chunks, an even number of them, is two half-row stages, so each half's
// copy overlaps work on the other; other rows are one stage.  Rows of up to
// 448 x 4 chunks run two CTAs per SM, longer ones one CTA of up to 1024
// threads.
bool plan_silu_tma_token(int64_t T, int nch, int mode, int sms, SiluTmaPlan *out) {
  if (mode != VG_SCALE_PER_TOKEN || T < 2LL * sms || nch < 512) return false;
  SiluTmaPlan p;
  p.vpt = 4;
  p.nseg = (nch >= 1024 && nch % 2 == 0) ? 2 : 1;
  p.block = ((nch / p.nseg + p.vpt / p.nseg - 1) / (p.vpt / p.nseg) + 31) / 32 * 32;
  const size_t smem = silu_tma_token_smem_bytes(nch * 8, p.nseg);
  if (smem > kTmaMaxSmem - 1024 || p.block > 1024) return false;
  const int ctas = (p.block <= 512 && 2 * smem <= 220 * 1024) ? 2 : 1;
  p.grid = T < (int64_t)sms * ctas ? T : (int64_t)sms * ctas;
  p.smem = cap_residency_smem(ctas, smem);
  *out = p;
  return true;
}

// The persistent TMA kernel pays off for dynamic scales once every SM has
// several rows to stream: it needs T >= 4 rows per SM and a row whose
// two-stage ring fits in shared memory.  Measured on GB300 over H = 2048..8192
// and T = 2048..32768: about 384 resident threads per SM with two stages per
// CTA stream best.  Fewer threads leave the SM short of warps; more CTAs or
// deeper rings keep more row copies in flight across the GPU than the memory
// system serves well, and run slower.  When a CTA would get fewer than ten
// rows, one more CTA of 128 threads or more evens out the tail.
bool plan_norm_tma(int64_t T, int H, bool res, int mode, int ngroups, int sms, TmaPlan *out) {
  const int nch = H / 8;
  // static scales gain nothing from staging: the register kernel already
  // streams at the copy roofline there
  if (mode == VG_SCALE_STATIC || T < 4LL * sms || nch < 256) return false;
  TmaPlan p;
  p.vpt = 4;
  while (p.vpt < 8 && (nch + p.vpt - 1) / p.vpt > 256) p.vpt *= 2;
  p.block = ((nch + p.vpt - 1) / p.vpt + 31) / 32 * 32;
  p.stages = 2;
  const int slots = mode == VG_SCALE_PER_TOKEN ? 1 : ngroups;
  const size_t bytes = norm_tma_smem_bytes(H, res, p.stages, p.block, p.vpt, slots);
  if (bytes > kTmaMaxSmem) return false;
  int ctas = (384 + p.block - 1) / p.block;
  if (p.block >= 128 && T < 10LL * sms * ctas) ++ctas;
  while (ctas > 1 && (bytes * ctas > 220 * 1024 || ctas * p.block > 1024)) --ctas;
  p.grid = T < (int64_t)sms * ctas ? T : (int64_t)sms * ctas;
  p.smem = cap_residency_smem(ctas, bytes);
  *out = p;
  return true;
}

// MLA dual norm.  Many tokens whose two rows fit eight chunks per lane of a
// warp (DeepSeek's 1536 + 512 exactly): one warp per token, eight warps per
// CTA -- the fewest instructions per element, but about 6 us of latency per
// token, so it pays from about 13 tokens per SM (measured: from T ~ 2048 on
// 152 SMs).  Otherwise a token's rows spread over a warp group: one token
// per CTA and one chunk per thread for few tokens (the shortest chain); two
// chunks per thread and tokens packed into CTAs of up to 512 threads for
// more.  A token's group stays within 512 threads up to four chunks per
// thread (eight allow 1024).
MlaPlan plan_mla(int64_t T, int nq, int nkv, bool q_fp8, int sms) {
  MlaPlan p;
  if ((nq + 31) / 32 + (nkv + 31) / 32 <= 8 && T >= 13LL * sms) {
    // DeepSeek's widths have instances with the token's chunks staged in
    // shared memory (five CTAs per SM); other widths hold them in registers
    // (four CTAs per SM).  Measured on GB300, staged against registers:
    // bf16 0.71 -> 0.81 (T = 8192), 0.89 -> 0.99 (32768); fp8 0.68 -> 0.71
    // (32768).
    const bool fixed = nq == 6 * 32 && nkv == 2 * 32;
    p.vpt = 0;
    p.thr[0] = p.thr[1] = 0;
    p.rpc = 8;
    p.block = 256;
    p.grid = (T + 7) / 8;
    // Up to one full wave, consecutive 8-token CTAs would leave some SMs a
    // whole CTA more than others (4096 tokens: 32 on 56 SMs, 24 on the
    // rest); instead every resident CTA slot gets a CTA and the tokens are
    // dealt out across them, warp by warp (at most one token apart per CTA).
    // Every CTA of such a wave prefetches its tokens into L2.  Measured on
    // GB300: T = 4096 bf16 0.54 -> 0.67, fp8 0.50 -> 0.53; T = 2048 bf16
    // 0.47 -> 0.48, fp8 0.33 -> 0.39.
    const int64_t wave = (int64_t)sms * (fixed ? 5 : 4);
    if (T < 8 * wave) {
      p.spread = true;
      p.grid = wave;
    }
    return p;
  }
  p.vpt = T >= 4LL * sms ? 2 : 1;
  auto threads = [&](int nch) { return ((nch + p.vpt - 1) / p.vpt + 31) / 32 * 32; };
  while (p.vpt < 8 && threads(nq) + threads(nkv) > 512) p.vpt *= 2;
  p.thr[0] = threads(nq);
  p.thr[1] = threads(nkv);
  const int per_tok = p.thr[0] + p.thr[1];
  p.rpc = T >= 2LL * sms ? (512 / per_tok > 1 ? 512 / per_tok : 1) : 1;
  if (p.rpc > 16) p.rpc = 16;
  p.block = p.rpc * per_tok;
  p.grid = (T + p.rpc - 1) / p.rpc;
  return p;
}

namespace {

vg_status mla_dual_norm(uint16_t *q_out, uint8_t *q_fp8, float *q_scale, uint16_t *kv_out,
                        const uint16_t *q_c, int64_t q_stride, const uint16_t *q_weight,
                        const uint16_t *kv_c, int64_t kv_stride, const uint16_t *kv_weight,
                        int64_t T, int64_t q_dim, int64_t kv_dim, float eps_q, float eps_kv,
                        vg_stream_t stream) {
  const bool fp8 = q_fp8 != nullptr || q_scale != nullptr;
  auto bad_dim = [](int64_t n, int64_t stride) {
    return n < 8 || n % 8 != 0 || n > VG_MAX_ROW || stride < n || stride % 8 != 0;
  };
  if (T < 0 || T > INT32_MAX || bad_dim(q_dim, q_stride) || bad_dim(kv_dim, kv_stride))
    return VG_ERR_BAD_SHAPE;
  if (T == 0) return VG_OK;
  if (!kv_out || !q_c || !q_weight || !kv_c || !kv_weight || (fp8 ? !q_fp8 || !q_scale : !q_out))
    return VG_ERR_NULL_PTR;
  if (misaligned(q_out, 16) || misaligned(q_fp8, 16) || misaligned(kv_out, 16) ||
      misaligned(q_c, 16) || misaligned(q_weight, 16) || misaligned(kv_c, 16) ||
      misaligned(kv_weight, 16) || misaligned(q_scale, 4))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  vg_status st = check_device(&sms);
  if (st != VG_OK) return st;
  clear_stale_error();

  MlaArgs a{};
  a.pf_ctas = 2 * sms;
  a.src[0] = q_c;
  a.src[1] = kv_c;
  a.w[0] = q_weight;
  a.w[1] = kv_weight;
  a.stride[0] = q_stride;
  a.stride[1] = kv_stride;
  a.out[0] = q_out;
  a.out[1] = kv_out;
  a.q8 = q_fp8;
  a.q_scale = q_scale;
  a.T = T;
  a.nch[0] = (int32_t)(q_dim / 8);
  a.nch[1] = (int32_t)(kv_dim / 8);
  a.eps[0] = eps_q;
  a.eps[1] = eps_kv;
  a.n[0] = (float)q_dim;
  a.n[1] = (float)kv_dim;
  a.inv_n[0] = 1.0f / (float)q_dim;
  a.inv_n[1] = 1.0f / (float)kv_dim;
  const MlaPlan p = plan_mla(T, a.nch[0], a.nch[1], fp8, sms);
  if (p.spread) a.pf_ctas = (int32_t)p.grid;  // a single wave: every CTA prefetches
  return launch_mla_dual_norm(a, fp8, p, (cudaStream_t)stream) == cudaSuccess ? VG_OK
                                                                               : VG_ERR_CUDA;
}

}  // namespace

}  // namespace vg

extern "C" {

vg_status vg_fused_mla_dual_rms_norm(uint16_t *q_out, uint16_t *kv_out, const uint16_t *q_c,
                                     int64_t q_stride, const uint16_t *q_weight,
                                     const uint16_t *kv_c, int64_t kv_stride,
                                     const uint16_t *kv_weight, int64_t num_tokens,
                                     int64_t q_dim, int64_t kv_dim, float eps_q,
                                     float eps_kv, vg_stream_t stream) {
  if (num_tokens > 0 && !q_out) return VG_ERR_NULL_PTR;
  return vg::mla_dual_norm(q_out, nullptr, nullptr, kv_out, q_c, q_stride, q_weight, kv_c,
                           kv_stride, kv_weight, num_tokens, q_dim, kv_dim, eps_q, eps_kv,
                           stream);
}

vg_status vg_fused_mla_dual_rms_norm_per_token_quant(
    uint8_t *q_fp8, float *q_scale, uint16_t *kv_out, const uint16_t *q_c, int64_t q_stride,
    const uint16_t *q_weight, const uint16_t *kv_c, int64_t kv_stride, const uint16_t *kv_weight,
    int64_t num_tokens, int64_t q_dim, int64_t kv_dim, float eps_q, float eps_kv,
    vg_stream_t stream) {
  if (num_tokens > 0 && (!q_fp8 || !q_scale)) return VG_ERR_NULL_PTR;
  return vg::mla_dual_norm(nullptr, q_fp8, q_scale, kv_out, q_c, q_stride, q_weight, kv_c,
                           kv_stride, kv_weight, num_tokens, q_dim, kv_dim, eps_q, eps_kv,
                           stream);
}

vg_status vg_fused_add_rms_norm_fp8(uint8_t *q, uint16_t *residual_out, float *scale,
                                    const uint16_t *x, const uint16_t *residual,
                                    const uint16_t *weight, int64_t num_tokens, int64_t hidden,
                                    float eps, int32_t mode, int32_t group_size,
                                    vg_stream_t stream) {
  vg_status st = vg::check_row(num_tokens, hidden, mode, group_size);
  const int32_t mode_flags = mode;
  mode &= 0xFF;
  if (st != VG_OK || num_tokens == 0) return st;
  if (!q || !scale || !x || !weight || ((residual == nullptr) != (residual_out == nullptr)))
    return VG_ERR_NULL_PTR;
  if (vg::misaligned(q, 16) || vg::misaligned(x, 16) || vg::misaligned(weight, 16) ||
      vg::misaligned(residual, 16) || vg::misaligned(residual_out, 16) || vg::misaligned(scale, 4))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  if ((st = vg::check_device(&sms)) != VG_OK) return st;
  vg::clear_stale_error();

  vg::NormArgs a{};
  a.pf_ctas = 2 * sms;
  a.q = q;
  a.res_out = residual_out;
  a.scale = scale;
  a.x = x;
  a.res = residual;
  a.w = weight;
  a.T = num_tokens;
  a.H = (int32_t)hidden;
  a.nch = (int32_t)(hidden / 8);
  a.gch = mode == VG_SCALE_PER_GROUP ? group_size / 8 : 1;
  a.ngroups = mode == VG_SCALE_PER_GROUP ? (int32_t)(hidden / group_size) : 1;
  a.eps = eps;
  a.inv_h = 1.0f / (float)hidden;
  vg::set_scale_layout(a, mode_flags, num_tokens);
  vg::TmaPlan tp;
  if (vg::plan_norm_tma(num_tokens, (int)hidden, residual != nullptr, mode, a.ngroups, sms, &tp))
    return vg::launch_norm_fp8_tma(a, mode, tp, (cudaStream_t)stream) == cudaSuccess ? VG_OK
                                                                                     : VG_ERR_CUDA;
  // Two chunks a thread in both scale modes (measured on GB300 for dynamic
  // scales at 2-4 rows per SM: 6-7 % faster than four chunks a thread).
  const vg::RowPlan plan = vg::plan_rows(num_tokens, a.nch, 2, sms);
  return vg::launch_norm_fp8(a, mode, plan, (cudaStream_t)stream) == cudaSuccess ? VG_OK
                                                                                   : VG_ERR_CUDA;
}

vg_status vg_fused_add_rms_norm_nvfp4(uint8_t *q4, uint8_t *block_scale, uint16_t *residual_out,
                                      const uint16_t *x, const uint16_t *residual,
                                      const uint16_t *weight, const float *global_scale,
                                      int64_t num_tokens, int64_t hidden, float eps,
                                      vg_stream_t stream) {
  vg_status st = vg::check_row(num_tokens, hidden, VG_SCALE_PER_TOKEN, 0);
  if (st != VG_OK) return st;
  if (hidden % 16 != 0) return VG_ERR_BAD_SHAPE;
  if (num_tokens == 0) return VG_OK;
  if (!q4 || !block_scale || !x || !weight || !global_scale ||
      ((residual == nullptr) != (residual_out == nullptr)))
    return VG_ERR_NULL_PTR;
  if (vg::misaligned(q4, 16) || vg::misaligned(x, 16) || vg::misaligned(weight, 16) ||
      vg::misaligned(residual, 16) || vg::misaligned(residual_out, 16) ||
      vg::misaligned(global_scale, 4))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  if ((st = vg::check_device(&sms)) != VG_OK) return st;
  vg::clear_stale_error();

  vg::NormArgs a{};
  a.pf_ctas = 2 * sms;
  a.q = q4;
  a.sf8 = block_scale;
  a.res_out = residual_out;
  a.scale = const_cast<float *>(global_scale);  // read only in this mode
  a.x = x;
  a.res = residual;
  a.w = weight;
  a.T = num_tokens;
  a.H = (int32_t)hidden;
  a.nch = (int32_t)(hidden / 8);
  a.gch = 2;
  a.ngroups = (int32_t)(hidden / 16);
  a.eps = eps;
  a.inv_h = 1.0f / (float)hidden;
  vg::set_scale_layout(a, VG_SCALE_PER_TOKEN, num_tokens);
  // the dynamic norm's plans; the block scales take half a DynScale each
  vg::TmaPlan tp;
  if (vg::plan_norm_tma(num_tokens, (int)hidden, residual != nullptr, vg::kNvfp4,
                        (a.ngroups + 1) / 2, sms, &tp))
    return vg::launch_norm_fp8_tma(a, vg::kNvfp4, tp, (cudaStream_t)stream) == cudaSuccess
               ? VG_OK
               : VG_ERR_CUDA;
  const vg::RowPlan plan = vg::plan_rows(num_tokens, a.nch, 4, sms);
  return vg::launch_norm_fp8(a, vg::kNvfp4, plan, (cudaStream_t)stream) == cudaSuccess
             ? VG_OK
             : VG_ERR_CUDA;
}

vg_status vg_fused_add_rms_norm_pad(uint16_t *out, uint16_t *residual_out, const uint16_t *x,
                                    const uint16_t *residual, const uint16_t *weight,
                                    int64_t num_tokens, int64_t hidden, int64_t padded_hidden,
                                    float eps, vg_stream_t stream) {
  vg_status st = vg::check_row(num_tokens, hidden, VG_SCALE_PER_TOKEN, 0);
  if (st != VG_OK) return st;
  if (padded_hidden < hidden || padded_hidden % 8 != 0 || padded_hidden > 2LL * VG_MAX_ROW)
    return VG_ERR_BAD_SHAPE;
  if (num_tokens == 0) return VG_OK;
  if (!out || !x || !weight || ((residual == nullptr) != (residual_out == nullptr)))
    return VG_ERR_NULL_PTR;
  if (vg::misaligned(out, 16) || vg::misaligned(x, 16) || vg::misaligned(weight, 16) ||
      vg::misaligned(residual, 16) || vg::misaligned(residual_out, 16))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  if ((st = vg::check_device(&sms)) != VG_OK) return st;
  vg::clear_stale_error();

  vg::NormArgs a{};
  a.pf_ctas = 2 * sms;
  a.res_out = residual_out;
  a.x = x;
  a.res = residual;
  a.w = weight;
  a.T = num_tokens;
  a.H = (int32_t)hidden;
  a.nch = (int32_t)(hidden / 8);
  a.gch = 1;
  a.ngroups = 1;
  a.eps = eps;
  a.inv_h = 1.0f / (float)hidden;
  a.out16 = out;
  a.nch_pad = (int32_t)(padded_hidden / 8);
  vg::set_scale_layout(a, VG_SCALE_PER_TOKEN, num_tokens);
  // the same plans as the dynamic per-token norm: one double-float inv per row
  vg::TmaPlan tp;
  if (vg::plan_norm_tma(num_tokens, (int)hidden, residual != nullptr, VG_SCALE_PER_TOKEN, 1, sms,
                        &tp))
    return vg::launch_norm_fp8_tma(a, vg::kBf16Pad, tp, (cudaStream_t)stream) == cudaSuccess
               ? VG_OK
               : VG_ERR_CUDA;
  const vg::RowPlan plan = vg::plan_rows(num_tokens, a.nch, 4, sms);
  return vg::launch_norm_fp8(a, vg::kBf16Pad, plan, (cudaStream_t)stream) == cudaSuccess
             ? VG_OK
             : VG_ERR_CUDA;
}

vg_status vg_fused_qk_norm_rope(uint16_t *qkv, const uint16_t *q_weight, const uint16_t *k_weight,
                                const float *cos_sin_cache, const int64_t *positions,
                                int64_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int64_t max_position, float eps, int32_t is_neox,
                                vg_stream_t stream) {
  if (num_tokens < 0 || num_tokens > INT32_MAX || num_q_heads < 0 || num_kv_heads < 0 ||
      num_q_heads + num_kv_heads < 1 || num_q_heads + 2LL * num_kv_heads > 4096 ||
      (head_dim != 64 && head_dim != 128 && head_dim != 256) || max_position < 1)
    return VG_ERR_BAD_SHAPE;
  if (num_tokens == 0) return VG_OK;
  if (!qkv || !cos_sin_cache || !positions || (num_q_heads > 0 && !q_weight) ||
      (num_kv_heads > 0 && !k_weight))
    return VG_ERR_NULL_PTR;
  if (vg::misaligned(qkv, 16) || vg::misaligned(q_weight, 16) || vg::misaligned(k_weight, 16) ||
      vg::misaligned(cos_sin_cache, 16) || vg::misaligned(positions, 8))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  vg_status st = vg::check_device(&sms);
  if (st != VG_OK) return st;
  vg::clear_stale_error();

  vg::QkArgs a{};
  a.pf_ctas = 2 * sms;
  a.qkv = qkv;
  a.qw = q_weight;
  a.kw = k_weight;
  a.cache = cos_sin_cache;
  a.pos = positions;
  a.T = num_tokens;
  a.row = (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim;
  a.max_pos = max_position;
  a.nh = num_q_heads + num_kv_heads;
  a.hq = num_q_heads;
  a.eps = eps;
  return vg::launch_qk_norm_rope(a, head_dim, is_neox != 0, (cudaStream_t)stream) == cudaSuccess
             ? VG_OK
             : VG_ERR_CUDA;
}

vg_status vg_silu_mul_fp8(uint8_t *q, float *scale, const uint16_t *gate_up, int64_t num_tokens,
                          int64_t inter, int32_t mode, int32_t group_size, vg_stream_t stream) {
  vg_status st = vg::check_row(num_tokens, inter, mode, group_size);
  const int32_t mode_flags = mode;
  mode &= 0xFF;
  if (st != VG_OK || num_tokens == 0) return st;
  if (!q || !scale || !gate_up) return VG_ERR_NULL_PTR;
  if (vg::misaligned(q, 16) || vg::misaligned(gate_up, 16) || vg::misaligned(scale, 4))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  if ((st = vg::check_device(&sms)) != VG_OK) return st;
  vg::clear_stale_error();

  vg::SiluArgs a{};
  a.pf_ctas = 2 * sms;
  a.q = q;
  a.scale = scale;
  a.gate_up = gate_up;
  a.T = num_tokens;
  a.I = (int32_t)inter;
  a.nch = (int32_t)(inter / 8);
  a.gch = mode == VG_SCALE_PER_GROUP ? group_size / 8 : 1;
  a.ngroups = mode == VG_SCALE_PER_GROUP ? (int32_t)(inter / group_size) : 1;
  vg::set_scale_layout(a, mode_flags, num_tokens);
  vg::SiluTmaPlan tp;
  if (vg::plan_silu_tma_token(num_tokens, a.nch, mode, sms, &tp))
    return vg::launch_silu_fp8_tma_token(a, tp, (cudaStream_t)stream) == cudaSuccess ? VG_OK
                                                                                    : VG_ERR_CUDA;
  const vg::RowPlan plan = vg::plan_silu(num_tokens, a.nch, mode, sms);
  return vg::launch_silu_fp8(a, mode, plan, (cudaStream_t)stream) == cudaSuccess ? VG_OK
                                                                                 : VG_ERR_CUDA;
}

vg_status vg_silu_mul_nvfp4(uint8_t *q4, uint8_t *block_scale, const uint16_t *gate_up,
                            const float *global_scale, int64_t num_tokens, int64_t inter,
                            vg_stream_t stream) {
  vg_status st = vg::check_row(num_tokens, inter, VG_SCALE_PER_TOKEN, 0);
  if (st != VG_OK) return st;
  if (inter % 16 != 0) return VG_ERR_BAD_SHAPE;
  if (num_tokens == 0) return VG_OK;
  if (!q4 || !block_scale || !gate_up || !global_scale) return VG_ERR_NULL_PTR;
  if (vg::misaligned(q4, 16) || vg::misaligned(gate_up, 16) || vg::misaligned(global_scale, 4))
    return VG_ERR_MISALIGNED;
  int sms = 0;
  if ((st = vg::check_device(&sms)) != VG_OK) return st;
  vg::clear_stale_error();

  vg::SiluArgs a{};
  a.pf_ctas = 2 * sms;
  a.q = q4;
  a.sf8 = block_scale;
  a.scale = const_cast<float *>(global_scale);  // read only in this mode
  a.gate_up = gate_up;
  a.T = num_tokens;
  a.I = (int32_t)inter;
  a.nch = (int32_t)(inter / 8);
  a.gch = 2;
  a.ngroups = (int32_t)(inter / 16);
  vg::set_scale_layout(a, VG_SCALE_PER_TOKEN, num_tokens);
  // no row state: the per-group plan (column segments, two chunks a thread)
  const vg::RowPlan plan = vg::plan_silu(num_tokens, a.nch, VG_SCALE_PER_GROUP, sms);
  return vg::launch_silu_fp8(a, vg::kNvfp4, plan, (cudaStream_t)stream) == cudaSuccess
             ? VG_OK
             : VG_ERR_CUDA;
}

vg_status vg_device_status(uint32_t *flags, int32_t reset) {
  if (!flags) return VG_ERR_NULL_PTR;
  const uint32_t v = vg::read_norm_status(reset != 0), w = vg::read_silu_status(reset != 0),
                 r = vg::read_rope_status(reset != 0), m = vg::read_mla_status(reset != 0);
  if (v == 0xFFFFFFFFu || w == 0xFFFFFFFFu || r == 0xFFFFFFFFu || m == 0xFFFFFFFFu)
    return VG_ERR_CUDA;
  *flags = v | w | r | m;
  return VG_OK;
}

const char *vg_status_string(vg_status s) {
  switch (s) {
    case VG_OK: return "ok";
    case VG_ERR_NULL_PTR: return "a required pointer is NULL (or residual/residual_out not paired)";
    case VG_ERR_BAD_SHAPE: return "bad shape: num_tokens < 0 or row length not a multiple of 8 in [8, VG_MAX_ROW]";
    case VG_ERR_MISALIGNED: return "misaligned pointer: tensors need 16-byte, scale 4-byte alignment";
    case VG_ERR_BAD_MODE: return "unknown scale mode";
    case VG_ERR_BAD_GROUP: return "per-group mode needs group_size 64 or 128 dividing the row length";
    case VG_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300)";
    case VG_ERR_CUDA: return "CUDA runtime or launch error";
  }
  return "unknown status";
}

int32_t vg_abi_version(void) { return VG_ABI_VERSION; }

}  // extern "C"
