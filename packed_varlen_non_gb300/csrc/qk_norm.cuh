// Per-row arithmetic of the q/k prologue: RMSNorm with gain, then the rot96
// rotation (NeoX pairs j <-> j+48 on dims 0..95, dims 96..127 unrotated).
//
// Pages: "h3-spark" model card, "What this config does" (Q RMSNorm + rot96
// RoPE fused into one kernel); vllm.cpp PR #26 "feat(minimax-h3)", "The
// device-resident forward (W2b)" (plain NeoX rotate_half fed by a per-row
// cos/sin cache; f32 reductions on the device).
//
// Every rounding is explicit (no contraction left to the compiler), so the
// separate prologue kernel (16 lanes per row) and the forward's fused Q path
// (one thread per row) produce bit-identical bf16 rows:
//   - the row is 16 chunks of 8 dims; a chunk's sum of squares is a
//     sequential fma chain from 0 over its 8 dims;
//   - the 16 chunk sums combine in a fixed tree: s1_k = p_k + p_{k+8},
//     s2_k = s1_k + s1_{k+4}, s3_k = s2_k + s2_{k+2}, total = s3_0 + s3_1
//     (a 16-lane xor butterfly with offsets 8, 4, 2, 1 gives exactly this
//     value in every lane, since fp addition commutes);
//   - r = rsqrt(total / 128 + eps); y = (x r) g; then
//     out_j = y_j c - y_{j+48} s and out_{j+48} = y_{j+48} c + y_j s.
#pragma once

#include "h3attn_internal.h"

namespace h3 {
namespace qkn {

__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
  return make_uint4(pack2(y[0], y[1]), pack2(y[2], y[3]), pack2(y[4], y[5]), pack2(y[6], y[7]));
}

// Sum of squares of one 8-dim chunk.
__device__ __forceinline__ float chunk_ss(const float (&x)[8]) {
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = __fmaf_rn(x[e], x[e], ss);
  return ss;
}

// The 16 chunk sums of a row, combined in the fixed tree.
__device__ __forceinline__ float tree16(const float (&p)[16]) {
  float s1[8], s2[4];
#pragma unroll
  for (int k = 0; k < 8; ++k) s1[k] = __fadd_rn(p[k], p[k + 8]);
#pragma unroll
  for (int k = 0; k < 4; ++k) s2[k] = __fadd_rn(s1[k], s1[k + 4]);
  return __fadd_rn(__fadd_rn(s2[0], s2[2]), __fadd_rn(s2[1], s2[3]));
}

__device__ __forceinline__ float inv_rms(float total, float eps) {
  return rsqrtf(__fmaf_rn(total, 1.0f / kHeadDim, eps));
}

__device__ __forceinline__ float scale_gain(float x, float r, float g) { return __fmul_rn(__fmul_rn(x, r), g); }

// dims j < 48 (partner j + 48) and dims j + 48 (partner j)
__device__ __forceinline__ float rot_lo(float y, float partner, float c, float s) {
  return __fmaf_rn(y, c, -__fmul_rn(partner, s));
}
__device__ __forceinline__ float rot_hi(float y, float partner, float c, float s) {
  return __fmaf_rn(y, c, __fmul_rn(partner, s));
}

// cos/sin of the 8 angles of lane lane16 of a 16-lane row group for token
// tok (lanes j and j + 6 share angles 8 (j % 6) .. + 8; lanes 12..15, the
// unrotated dims, get cos 1, sin 0).  rope: [S, 48] (cos, sin).
__device__ __forceinline__ void load_cs16(const float2* rope, int64_t tok, int lane16, float (&c)[8], float (&s)[8]) {
  if (lane16 < 12) {
    const float4* t = reinterpret_cast<const float4*>(rope + tok * kRopeHalf + (lane16 % 6) * 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 cs = __ldg(t + i);  // (cos, sin) of two consecutive angles
      c[2 * i] = cs.x;
      s[2 * i] = cs.y;
      c[2 * i + 1] = cs.z;
      s[2 * i + 1] = cs.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = 1.f;
      s[e] = 0.f;
    }
  }
}

// One row spread over 16 lanes (lane16 = lane within its group of 16, mask =
// the group's lanes): normalise x (this lane's 8 dims), apply the gain g (this
// lane's 8 gains) and the rotation.  c, s: cos/sin of this lane's 8 angles (1,
// 0 for lanes 12..15).
__device__ __forceinline__ void norm_rope16(float (&x)[8], const float (&g)[8], const float (&c)[8],
                                            const float (&s)[8], int lane16, unsigned mask, float eps) {
  float ss = chunk_ss(x);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(mask, ss, off, 16));
  const float r = inv_rms(ss, eps);
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = scale_gain(x[e], r, g[e]);
  const int partner = lane16 < 6 ? lane16 + 6 : (lane16 < 12 ? lane16 - 6 : lane16);
  float p[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = __shfl_sync(mask, y[e], partner, 16);
  if (lane16 < 6) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = rot_lo(y[e], p[e], c[e], s[e]);
  } else if (lane16 < 12) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = rot_hi(y[e], p[e], c[e], s[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = y[e];
  }
}

// The 8 gains of lane lane16 (gain: the head's 128 gains, 16-byte aligned).
__device__ __forceinline__ void load_gain16(const float* gain, int lane16, float (&g)[8]) {
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain + lane16 * 8));
  const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain + lane16 * 8 + 4));
  g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
  g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
}

}  // namespace qkn
}  // namespace h3
