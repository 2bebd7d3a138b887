// qk_norm_rope.cu -- per-head RMSNorm of Q and K, then the rotary embedding,
// in place, one pass over HBM.
//
// Implements "QK Norm + RoPE (enable_qk_norm_rope_fusion)" of the "Fusion
// torch.compile passes" page: split QKV -> per-head RMSNorm of the Q heads
// (q weight) and K heads (k weight) -> rotary embedding, as one kernel.  A
// qkv row is [Q heads | K heads | V heads], D columns a head; V is not
// touched.  The rotation reads an fp32 cos/sin cache [max_pos, D] (cos in
// the first D/2 columns, sin in the rest) at each token's position and
// turns the pairs (i, i + D/2) (neox) or (2i, 2i + 1) (gptj).
//
// Layout: one token per CTA (blockIdx.y splits very many heads); a head is
// D/8 chunks of 8 bf16 held by G = D/16 consecutive lanes, lane l holding
// chunks l and l + G -- so a neox pair (i, i + D/2) lives in one lane, and a
// gptj pair inside one chunk.  Each lane keeps t = x * w (exact in fp32).
//
// Arithmetic (fp32): the head's sum of squares in fp32 (longest path 11
// roundings of non-negative terms: <= 11u), inv = rsqrt(sum/D + eps)
// (<= 10u with rsqrtf's 2 ulps), o = t_a c -/+ t_b s by Kahan's FMA
// algorithm for a*c - b*s (q = b*s, e = fma(b, s, -q), f = fma(a, c, -q),
// o = f - e: within 2 ulps of the exact value even under cancellation), and
// p = o * inv rounded once to bf16.  So p is within ~15u (2^-20 relative) of
// the exact result, and its bf16 differs from the correctly rounded one only
// where the exact value lies that close to a bf16 midpoint, by one ulp.
#include "common.cuh"
#include "launch.h"
#include "row_norm.cuh"

namespace vg {

// Status word of this translation unit's kernels: kErrBadPosition when a
// position lies outside [0, max_pos) (that head is left as it was).
__device__ uint32_t g_rope_status;

namespace {

__device__ __forceinline__ void load8f(const float *p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load4f(const float *p, float (&v)[8], int at) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  v[at] = a.x; v[at + 1] = a.y; v[at + 2] = a.z; v[at + 3] = a.w;
}

// Two elements of a*c -/+ b*s (Kahan), packed; a zero keeps the plain
// expression's sign.  nb = -b for the minus form.
__device__ __forceinline__ float2 kahan2x(float2 a, float2 c, float2 nb, float2 s) {
  const float2 q = f2_mul(nb, s);
  const float2 e = f2_fma(nb, s, make_float2(-q.x, -q.y));
  const float2 f = f2_fma(a, c, q);
  const float2 o = f2_add(f, e);
  return make_float2(e.x != 0.f ? o.x : f.x, e.y != 0.f ? o.y : f.y);
}

template <int G, bool NEOX>
__global__ void __launch_bounds__(512) qk_norm_rope_kernel(const QkArgs a) {
  constexpr int D = G * 16;
  const int lane = threadIdx.x & 31;
  const int l = lane & (G - 1);
  const int64_t t = blockIdx.x;
  const int h = ((int)blockIdx.y * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5)) * (32 / G) + lane / G;
  // Launched with programmatic dependent launch: nothing in global memory
  // before the previous grid has finished, except that the CTA's heads are
  // asked into L2 first; the next grid may be scheduled once the loads are out.
  if (threadIdx.x == 0 && (int)blockIdx.x < a.pf_ctas) {
    const int h0 = (int)blockIdx.y * (int)(blockDim.x >> 5) * (32 / G);
    const int nh = a.nh - h0 < (int)(blockDim.x >> 5) * (32 / G) ? a.nh - h0 : (int)(blockDim.x >> 5) * (32 / G);
    prefetch_l2(a.qkv + t * a.row + (int64_t)h0 * D, 2u * (uint32_t)(nh * D));
  }
  pdl_wait();
  // The head's loads do not depend on the token's position, so they go out
  // together with it (a head with a bad position is loaded but not stored);
  // only the cos/sin row waits for the position.
  const bool in_head = h < a.nh;
  uint16_t *head = a.qkv + t * a.row + (in_head ? (int64_t)h * D : 0);
  const uint16_t *w = h < a.hq ? a.qw : a.kw;
  const int64_t pos = a.pos[t];
  // chunk 0 of the lane: l (first half of the head), chunk 1: l + G
  const uint4 xa = in_head ? ld_stream(head + l * kElemsPerChunk) : make_uint4(0, 0, 0, 0);
  const uint4 xb = in_head ? ld_stream(head + (l + G) * kElemsPerChunk) : make_uint4(0, 0, 0, 0);
  const uint4 wa = in_head ? ld_keep(w + l * kElemsPerChunk) : make_uint4(0, 0, 0, 0);
  const uint4 wb = in_head ? ld_keep(w + (l + G) * kElemsPerChunk) : make_uint4(0, 0, 0, 0);
  const bool live = in_head && pos >= 0 && pos < a.max_pos;  // same for the head's lanes
  if (in_head && !live && l == 0) atomicOr(&g_rope_status, kErrBadPosition);
  pdl_launch_dependents();
  float2 ta[4], tb[4];
  float cmax;
  RowAcc acc;
  pass1_chunk<false, false>(xa, xa, wa, ta, cmax, acc);
  pass1_chunk<false, false>(xb, xb, wb, tb, cmax, acc);
  float ss = acc.ss.x + acc.ss.y;
#pragma unroll
  for (int o = G >> 1; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float y = rsqrtf(fmaf(ss, 1.0f / (float)D, a.eps));

  // mine[0..7]: chunk 0, mine[8..15]: chunk 1; other: each element's pair
  // partner; c, s: its pair's cos and sin; submask bit k: minus sign
  float mine[16], other[16], c[16], s[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mine[2 * i] = ta[i].x;
    mine[2 * i + 1] = ta[i].y;
    mine[8 + 2 * i] = tb[i].x;
    mine[8 + 2 * i + 1] = tb[i].y;
  }
  const float *cs = a.cache + (live ? pos * D : 0);
  uint32_t submask;
  if (NEOX) {  // element k of chunk 0 pairs with element k of chunk 1: pair 8l + k
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      other[k] = mine[8 + k];
      other[8 + k] = mine[k];
    }
    float c8[8] = {}, s8[8] = {};
    if (live) {
      load8f(cs + 8 * l, c8);
      load8f(cs + D / 2 + 8 * l, s8);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      c[k] = c[8 + k] = c8[k];
      s[k] = s[8 + k] = s8[k];
    }
    submask = 0x00FFu;
  } else {  // pairs (2i, 2i + 1) inside each chunk: pair 4 chunk + k / 2
#pragma unroll
    for (int k = 0; k < 16; ++k) other[k] = mine[k ^ 1];
    float c4[8] = {}, s4[8] = {};
    if (live) {
      load4f(cs + 4 * l, c4, 0);
      load4f(cs + 4 * (l + G), c4, 4);
      load4f(cs + D / 2 + 4 * l, s4, 0);
      load4f(cs + D / 2 + 4 * (l + G), s4, 4);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      c[k] = c4[k >> 1];
      s[k] = s4[k >> 1];
    }
    submask = 0x5555u;
  }

  float p[16];
#pragma unroll
  for (int k = 0; k < 16; k += 2) {
    const bool m0 = (submask >> k) & 1u, m1 = (submask >> (k + 1)) & 1u;
    const float2 o = kahan2x(make_float2(mine[k], mine[k + 1]), make_float2(c[k], c[k + 1]),
                             make_float2(m0 ? -other[k] : other[k], m1 ? -other[k + 1] : other[k + 1]),
                             make_float2(s[k], s[k + 1]));
    const float2 pp = f2_mul(o, make_float2(y, y));
    p[k] = pp.x;
    p[k + 1] = pp.y;
  }
  const uint4 oa = make_uint4(pack_bf16x2_rn(p[0], p[1]), pack_bf16x2_rn(p[2], p[3]),
                              pack_bf16x2_rn(p[4], p[5]), pack_bf16x2_rn(p[6], p[7]));
  const uint4 ob = make_uint4(pack_bf16x2_rn(p[8], p[9]), pack_bf16x2_rn(p[10], p[11]),
                              pack_bf16x2_rn(p[12], p[13]), pack_bf16x2_rn(p[14], p[15]));
  [[maybe_unused]] const uint64_t bytes = VG_ROWS(a.T) * 2ull * (uint64_t)a.row;
  if (live && VG_ACCESS_OK(g_rope_status, head + l * kElemsPerChunk, 16, a.qkv, bytes))
    st_stream(head + l * kElemsPerChunk, oa);
  if (live && VG_ACCESS_OK(g_rope_status, head + (l + G) * kElemsPerChunk, 16, a.qkv, bytes))
    st_stream(head + (l + G) * kElemsPerChunk, ob);
}

// One token per CTA: up to 16 warps of heads; blockIdx.y covers the rest.
template <int G>
cudaError_t launch_g(const QkArgs &a, bool neox, cudaStream_t s) {
  const int heads_per_warp = 32 / G;
  int warps = (a.nh + heads_per_warp - 1) / heads_per_warp;
  if (warps > 16) warps = 16;
  const dim3 grid((unsigned)a.T, (unsigned)((a.nh + warps * heads_per_warp - 1) / (warps * heads_per_warp)));
  return neox ? launch_pdl(qk_norm_rope_kernel<G, true>, grid, dim3(warps * 32), 0, s, a)
              : launch_pdl(qk_norm_rope_kernel<G, false>, grid, dim3(warps * 32), 0, s, a);
}

}  // namespace

cudaError_t launch_qk_norm_rope(const QkArgs &a, int head_dim, bool neox, cudaStream_t s) {
  switch (head_dim) {
    case 64: return launch_g<4>(a, neox, s);
    case 128: return launch_g<8>(a, neox, s);
    default: return launch_g<16>(a, neox, s);
  }
}

uint32_t read_rope_status(bool reset) {
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_rope_status, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (reset) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_rope_status, &zero, sizeof(zero)) != cudaSuccess) return 0xFFFFFFFFu;
  }
  return v;
}

}  // namespace vg
