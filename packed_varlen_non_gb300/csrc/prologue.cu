// The q/k prologue kernel: per-head RMSNorm with gain, then the 3D rotary
// embedding on dims 0..95 (NeoX pairs j <-> j+48, angles from the plan's
// per-row cos/sin table); dims 96..127 only take the norm.
//
// Pages: "h3-spark" model card, "What this config does" (Q RMSNorm + rot96
// RoPE fused into one kernel, byte-exact on default and non-default
// streams); vllm.cpp PR #26 "feat(minimax-h3)", "The device-resident forward
// (W2b)" (plain NeoX rotate_half fed by a per-row cos/sin cache; f32
// reductions on the device).
//
// HBM-bound: each (token, head) row of q and of k is read once (256 B) and
// written once.  Sixteen lanes own one row, eight dims (one 16-byte vector)
// each: lanes 0..5 hold dims 0..47, lanes 6..11 dims 48..95 (their rotation
// partners, six lanes apart), lanes 12..15 the pass-through dims 96..127.
// The sum of squares is a 16-lane butterfly; partners swap normalised values
// with one shuffle per dim.  A warp covers two consecutive (token, head) rows,
// 512 contiguous bytes when the heads of a token are contiguous.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "qk_norm.cuh"

namespace h3 {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 16;

// Normalise x (this lane's 8 dims of one row), apply gain and the rotation
// (the arithmetic of qk_norm.cuh, spread over 16 lanes).
__device__ __forceinline__ void norm_rope(float (&x)[8], const float* gain, const float (&c)[8],
                                          const float (&s)[8], int lane16, unsigned mask,
                                          float eps) {
  float ss = qkn::chunk_ss(x);
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(mask, ss, off, 16));
  const float r = qkn::inv_rms(ss, eps);
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gain + lane16 * 8));
  const float4 g1 = __ldg(reinterpret_cast<const float4*>(gain + lane16 * 8 + 4));
  const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = qkn::scale_gain(x[e], r, g[e]);
  const int partner = lane16 < 6 ? lane16 + 6 : (lane16 < 12 ? lane16 - 6 : lane16);
  float p[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = __shfl_sync(mask, y[e], partner, 16);
  if (lane16 < 6) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = qkn::rot_lo(y[e], p[e], c[e], s[e]);
  } else if (lane16 < 12) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = qkn::rot_hi(y[e], p[e], c[e], s[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = y[e];
  }
}

__global__ void __launch_bounds__(kThreads) qk_prologue_kernel(PrologueArgs a) {
  const int lane16 = threadIdx.x & 15;
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  const int64_t n_rows = a.S * a.H;
  const int64_t step = (int64_t)gridDim.x * kRowsPerBlock;
  const __nv_bfloat16* qi = static_cast<const __nv_bfloat16*>(a.q_in);
  const __nv_bfloat16* ki = static_cast<const __nv_bfloat16*>(a.k_in);
  __nv_bfloat16* qo = static_cast<__nv_bfloat16*>(a.q_out);
  __nv_bfloat16* ko = static_cast<__nv_bfloat16*>(a.k_out);
  const bool with_q = a.q_in != nullptr;  // k only when q is handled by the forward
#pragma unroll 1
  for (int64_t row = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 4); row < n_rows;
       row += step) {
    const int64_t tok = row / a.H;
    const int head = (int)(row - tok * a.H);
    const int64_t in_off = tok * a.in_stride + head * kHeadDim + lane16 * 8;
    const uint4 kraw = __ldcs(reinterpret_cast<const uint4*>(ki + in_off));
    const uint4 qraw = with_q ? __ldcs(reinterpret_cast<const uint4*>(qi + in_off)) : make_uint4(0, 0, 0, 0);
    float c[8], s[8];
    if (lane16 < 12) {
      const float4* t =
          reinterpret_cast<const float4*>(a.rope + tok * kRopeHalf + (lane16 % 6) * 8);
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
    float xk[8];
    qkn::unpack8(kraw, xk);
    norm_rope(xk, a.gain_k + head * a.gain_head_stride, c, s, lane16, mask, a.eps);
    const int64_t out_off = tok * a.out_stride + head * kHeadDim + lane16 * 8;
    __stcs(reinterpret_cast<uint4*>(ko + out_off), qkn::pack8(xk));
    if (with_q) {
      float xq[8];
      qkn::unpack8(qraw, xq);
      norm_rope(xq, a.gain_q + head * a.gain_head_stride, c, s, lane16, mask, a.eps);
      __stcs(reinterpret_cast<uint4*>(qo + out_off), qkn::pack8(xq));
    }
  }
}

}  // namespace

cudaError_t launch_qk_prologue(const PrologueArgs& a, int num_sms, cudaStream_t stream) {
  const int64_t n_rows = a.S * a.H;
  if (n_rows == 0) return cudaSuccess;
  // 8 blocks of 256 threads per SM (at 64 registers, 4 of them are resident at
  // a time; the grid-stride loop keeps the rest queued behind), or fewer
  // when there is less work.  A variant with two rows of loads in flight per
  // lane group and a single resident wave measured slower (3.7 vs 4.4 TB/s).
  const int64_t want = (n_rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t full = (int64_t)num_sms * 8;
  const int grid = (int)(want < full ? want : full);
  qk_prologue_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace h3
