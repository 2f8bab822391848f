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

__global__ void __launch_bounds__(kThreads, 4) qk_prologue_kernel(PrologueArgs a) {
  const int lane16 = threadIdx.x & 15;
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  const int64_t n_rows = a.S * a.H;
  const int64_t step = (int64_t)gridDim.x * kRowsPerBlock;
  const __nv_bfloat16* qi = static_cast<const __nv_bfloat16*>(a.q_in);
  const __nv_bfloat16* ki = static_cast<const __nv_bfloat16*>(a.k_in);
  __nv_bfloat16* qo = static_cast<__nv_bfloat16*>(a.q_out);
  __nv_bfloat16* ko = static_cast<__nv_bfloat16*>(a.k_out);
  const bool with_q = a.q_in != nullptr;  // k only when q is handled by the forward
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 4);
  if (row0 >= n_rows) return;  // the whole 16-lane group, which alone shuffles together
  // The launcher makes the grid-stride step a multiple of H (or gives each
  // lane group one row), so a lane group keeps one head and loads its gains once.
  const int head = (int)(row0 % a.H);
  float gk[8], gq[8];
  qkn::load_gain16(a.gain_k + head * a.gain_head_stride, lane16, gk);
  if (with_q) qkn::load_gain16(a.gain_q + head * a.gain_head_stride, lane16, gq);
#pragma unroll 1
  for (int64_t row = row0; row < n_rows; row += step) {
    const int64_t tok = row / a.H;
    const int64_t in_off = tok * a.in_stride + head * kHeadDim + lane16 * 8;
    const uint4 kraw = __ldcs(reinterpret_cast<const uint4*>(ki + in_off));
    const uint4 qraw = with_q ? __ldcs(reinterpret_cast<const uint4*>(qi + in_off)) : make_uint4(0, 0, 0, 0);
    float c[8], s[8];
    qkn::load_cs16(a.rope, tok, lane16, c, s);
    float xk[8];
    qkn::unpack8(kraw, xk);
    qkn::norm_rope16(xk, gk, c, s, lane16, mask, a.eps);
    const int64_t out_off = tok * a.out_stride + head * kHeadDim + lane16 * 8;
    __stcs(reinterpret_cast<uint4*>(ko + out_off), qkn::pack8(xk));
    if (with_q) {
      float xq[8];
      qkn::unpack8(qraw, xq);
      qkn::norm_rope16(xq, gq, c, s, lane16, mask, a.eps);
      __stcs(reinterpret_cast<uint4*>(qo + out_off), qkn::pack8(xq));
    }
  }
}

}  // namespace

cudaError_t launch_qk_prologue(const PrologueArgs& a, int num_sms, cudaStream_t stream) {
  const int64_t n_rows = a.S * a.H;
  if (n_rows == 0) return cudaSuccess;
  // 8 blocks of 256 threads per SM (capped at 64 registers, 4 of them are
  // resident at a time; the grid-stride loop keeps the rest queued behind), or
  // fewer when there is less work.  A variant with two rows of loads in flight
  // per lane group and a single resident wave measured slower (3.7 vs 4.4
  // TB/s); hoisting the gains at 72 registers (3 blocks resident) measured 112
  // instead of 94 us.
  // A full grid is rounded down to a multiple of H / gcd(16, H) blocks, so that
  // the grid-stride step (16 rows per block) is a multiple of H and a lane
  // group's head stays fixed.
  const int64_t want = (n_rows + kRowsPerBlock - 1) / kRowsPerBlock;
  int64_t full = (int64_t)num_sms * 8;
  int64_t g16 = kRowsPerBlock, h = a.H;
  while (h != 0) {
    const int64_t t = g16 % h;
    g16 = h;
    h = t;
  }
  const int64_t unit = a.H / g16;  // g16 = gcd(16, H)
  full = full / unit * unit;
  if (full < unit) full = unit;
  const int grid = (int)(want < full ? want : full);
  qk_prologue_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace h3
