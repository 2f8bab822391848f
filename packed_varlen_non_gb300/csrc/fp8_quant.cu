// Quantisation of the attention inputs to FP8 (e4m3) for the FP8 variant of
// the forward: q-hat per (token, head) row, k-hat per (head, 128-key tile of a
// document), v per (head, channel) over all tokens and written transposed
// (channel-major, keys contiguous, each document starting on a 16-key
// boundary so that a key tile's TMA coordinate is 16-byte aligned) for the PV
// product's K-major B operand.
//
// Pages: vllm.cpp PR #26 "feat(minimax-h3)" and the "h3-spark" model card,
// "What this config does" name a SageAttention2++-style INT8/FP8 attention
// without its scheme; this is the plainest scheme that runs both products on
// FP8 tensor cores.  Every decision is made in fp32 -- scale = amax / 448 and
// r = 448 / amax by correctly rounded divisions (both 1 for an all-zero row,
// tile or channel), code = e4m3(x * r) by one correctly rounded product and
// the hardware round-to-nearest-even conversion with saturation -- so the
// codes are the ones an fp32 reference computes.
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "qk_norm.cuh"

namespace h3 {

namespace {

constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ float fp8_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f; }
__device__ __forceinline__ float fp8_recip(float amax) { return amax > 0.f ? __fdiv_rn(kE4m3Max, amax) : 1.f; }

// two e4m3 codes, lo in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// 8 codes (one lane's 8 dims) as 8 bytes
__device__ __forceinline__ uint2 codes8(const float (&x)[8], float r) {
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = e4m3x2(__fmul_rn(x[2 * i], r), __fmul_rn(x[2 * i + 1], r));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// q-hat: 16 lanes per (token, head) row, 8 dims each; four rows per lane
// group per iteration, their loads issued together.
__global__ void __launch_bounds__(256) quant_rows_kernel(Fp8QuantArgs a) {
  const int lane16 = threadIdx.x & 15;
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  const int64_t n_rows = a.S * a.H;
  const int64_t stride = (int64_t)gridDim.x * 16;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.q_hat);
  uint8_t* out = static_cast<uint8_t*>(a.q8);
  for (int64_t row0 = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4); row0 < n_rows; row0 += 4 * stride) {
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t row = row0 + u * stride;
      if (row < n_rows) {
        const int64_t t = row / a.H;
        const int h = (int)(row - t * a.H);
        raw[u] = __ldg(reinterpret_cast<const uint4*>(x + t * a.stride + h * kHeadDim + lane16 * 8));
      } else {
        raw[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t row = row0 + u * stride;
      if (row >= n_rows) break;  // uniform across the lane group
      float f[8];
      unpack8(raw[u], f);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[e]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, off, 16));
      *reinterpret_cast<uint2*>(out + row * kHeadDim + lane16 * 8) = codes8(f, fp8_recip(m));
      if (lane16 == 0) {
        const int64_t t = row / a.H;
        a.sq[(int64_t)(row - t * a.H) * a.S + t] = fp8_scale(m);
      }
    }
  }
}

// k-hat: one block per (key tile, head); 16 lanes per token row (256
// contiguous bytes), so thread i takes dims [8 (i%16), +8) of tokens
// b + i/16, b + i/16 + 16, ... (eight of them).
__global__ void __launch_bounds__(256) quant_ktiles_kernel(Fp8QuantArgs a) {
  __shared__ float warp_max[8];
  const int tile = blockIdx.x, h = blockIdx.y;
  const int4 te = a.tiles[tile];
  const int tl0 = threadIdx.x >> 4, d0 = (threadIdx.x & 15) * 8;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.k_hat) + h * kHeadDim + d0;
  float f[8][8];
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int64_t t = te.x + tl0 + 16 * u;
    if (t < te.y) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(x + t * a.stride)), f[u]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[u][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(f[u][e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  m = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, warp_max[w]);
  const float r = fp8_recip(m), sc = fp8_scale(m);
  uint8_t* out = static_cast<uint8_t*>(a.k8) + h * kHeadDim + d0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int64_t t = te.x + tl0 + 16 * u;
    if (t < te.y) {
      *reinterpret_cast<uint2*>(out + t * a.H * kHeadDim) = codes8(f[u], r);
      if (d0 == 0) a.sk[(int64_t)h * a.S + t] = sc;
    }
  }
}

// The q/k prologue and the q/k quantisation in one pass (h3attn_qk_prologue_fp8):
// the prologue's RMSNorm + rot96 arithmetic (qk_norm.cuh), its bf16 rounding,
// then the codes and scales of quant_rows_kernel and quant_ktiles_kernel from
// those bf16 values -- the same bits as the three kernels in turn, without
// q-hat and k-hat going through HBM.  The block also folds its tile's v rows
// into the per-channel maxima (vmax_kernel's job).  One block per (key tile,
// head), 16 lanes per token row: thread i takes dims [8 (i%16), +8) of
// tokens b + i/16 + 16u (u < 8), four rows at a time whose q and k loads it
// issues together before working on them (80 registers: three blocks per SM).
// A q row is quantised as soon as it is normalised; the k rows wait in shared
// memory (bf16) until the tile's amax is known.
__global__ void __launch_bounds__(256, 3) prologue_quant_kernel(PrologueArgs p, Fp8QuantArgs a) {
  __shared__ uint4 k_tile[128][16];     // the tile's k-hat rows, bf16 (32 KB)
  __shared__ float warp_max[8];
  __shared__ float v_max[8][kHeadDim];  // per warp, per channel
  const int4 te = a.tiles[blockIdx.x];
  const int h = blockIdx.y;
  const int lane16 = threadIdx.x & 15, tl0 = threadIdx.x >> 4, warp = threadIdx.x >> 5;
  const unsigned mask = 0xffffu << (threadIdx.x & 16);
  const __nv_bfloat16* qi = static_cast<const __nv_bfloat16*>(p.q_in) + h * kHeadDim + lane16 * 8;
  const __nv_bfloat16* ki = static_cast<const __nv_bfloat16*>(p.k_in) + h * kHeadDim + lane16 * 8;
  const __nv_bfloat16* vi = static_cast<const __nv_bfloat16*>(a.v) + h * kHeadDim + lane16 * 8;
  const float* gqp = p.gain_q + h * p.gain_head_stride;
  const float* gkp = p.gain_k + h * p.gain_head_stride;
  uint8_t* q8 = static_cast<uint8_t*>(a.q8) + h * kHeadDim + lane16 * 8;
  // rows of this lane group: tokens te.x + tl0 + 16 u for u < n_rows
  const int rem = te.y - te.x - tl0;
  const int n_rows = rem > 0 ? (rem + 15) / 16 : 0;
  // Straight-line over each batch's rows (the next row's table loads can then
  // be issued early): a row past the tile end is all zeros, stays zero through
  // the norm and rotation (its table row is the tile's first), and is not
  // stored.
  float kmax = 0.f;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint4 kraw[4], qraw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = 4 * half + i;
      const int64_t t = te.x + tl0 + 16 * u;
      if (u < n_rows) {
        kraw[i] = __ldcs(reinterpret_cast<const uint4*>(ki + t * p.in_stride));
        qraw[i] = __ldcs(reinterpret_cast<const uint4*>(qi + t * p.in_stride));
      } else {
        kraw[i] = qraw[i] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = 4 * half + i;
      const bool valid = u < n_rows;
      const int64_t t = te.x + tl0 + 16 * u;
      float c[8], s[8];
      qkn::load_cs16(p.rope, valid ? t : (int64_t)te.x, lane16, c, s);
      float x[8];
      qkn::unpack8(kraw[i], x);
      float gk[8];
      qkn::load_gain16(gkp, lane16, gk);
      qkn::norm_rope16(x, gk, c, s, lane16, mask, p.eps);
      const uint4 kb = qkn::pack8(x);
      k_tile[tl0 + 16 * u][lane16] = kb;
      qkn::unpack8(kb, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) kmax = fmaxf(kmax, fabsf(x[e]));
      qkn::unpack8(qraw[i], x);
      float gq[8];
      qkn::load_gain16(gqp, lane16, gq);
      qkn::norm_rope16(x, gq, c, s, lane16, mask, p.eps);
      qkn::unpack8(qkn::pack8(x), x);
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(x[e]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, off, 16));
      if (valid) {
        *reinterpret_cast<uint2*>(q8 + t * a.H * kHeadDim) = codes8(x, fp8_recip(m));
        if (lane16 == 0) a.sq[(int64_t)h * a.S + t] = fp8_scale(m);
      }
    }
  }
  // v: this thread's channel maxima over its rows
  uint4 vraw[8];
#pragma unroll
  for (int u = 0; u < 8; ++u)
    vraw[u] = u < n_rows ? __ldcs(reinterpret_cast<const uint4*>(vi + (int64_t)(te.x + tl0 + 16 * u) * a.stride))
                         : make_uint4(0, 0, 0, 0);
  float vm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    float x[8];
    qkn::unpack8(vraw[u], x);
#pragma unroll
    for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], fabsf(x[e]));
  }
  // block maxima: k over the tile, v per channel (rows past the tile end count as 0)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
#pragma unroll
  for (int e = 0; e < 8; ++e) vm[e] = fmaxf(vm[e], __shfl_xor_sync(0xffffffffu, vm[e], 16));
  if ((threadIdx.x & 31) == 0) warp_max[warp] = kmax;
  if ((threadIdx.x & 16) == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v_max[warp][lane16 * 8 + e] = vm[e];
  }
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    float m = v_max[0][threadIdx.x];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, v_max[w][threadIdx.x]);
    // non-negative floats order like their bit patterns
    atomicMax(reinterpret_cast<uint32_t*>(a.sv) + h * kHeadDim + threadIdx.x, __float_as_uint(m));
  }
  float m = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, warp_max[w]);
  const float r = fp8_recip(m), sc = fp8_scale(m);
  uint8_t* k8 = static_cast<uint8_t*>(a.k8) + h * kHeadDim + lane16 * 8;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if (u >= n_rows) break;
    const int64_t t = te.x + tl0 + 16 * u;
    float x[8];
    qkn::unpack8(k_tile[tl0 + 16 * u][lane16], x);
    *reinterpret_cast<uint2*>(k8 + t * a.H * kHeadDim) = codes8(x, r);
    if (lane16 == 0) a.sk[(int64_t)h * a.S + t] = sc;
  }
}

// v, pass 1: per-(head, channel) amax over all tokens into the scale buffer's
// bits (non-negative floats order like their bit patterns).  Block (x, y):
// 128 groups of 8 channels from group 128 x, tokens [64 y, 64 y + 64);
// consecutive threads read consecutive 16 bytes of a token row.
constexpr int kVmaxTokens = 64;
__global__ void __launch_bounds__(128) vmax_kernel(Fp8QuantArgs a) {
  const int g = blockIdx.x * 128 + threadIdx.x;  // group of 8 channels
  if (g >= a.H * 16) return;
  const int h = g >> 4, c0 = (g & 15) * 8;
  const int64_t t0 = (int64_t)blockIdx.y * kVmaxTokens;
  const int64_t t1 = t0 + kVmaxTokens < a.S ? t0 + kVmaxTokens : a.S;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.v) + h * kHeadDim + c0;
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 16
  for (int64_t t = t0; t < t1; ++t) {
    float f[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(x + t * a.stride)), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = fmaxf(m[e], fabsf(f[e]));
  }
  uint32_t* bits = reinterpret_cast<uint32_t*>(a.sv) + h * kHeadDim + c0;
#pragma unroll
  for (int e = 0; e < 8; ++e) atomicMax(bits + e, __float_as_uint(m[e]));
}

// v, pass 2: codes, transposed through shared memory: one block per (key
// tile, head) writes v8t[h][c][vb .. vb + n) for all 128 channels, where the
// tile's n <= 128 keys start at vb in the transposed layout (every document
// starts on a 16-key boundary); a document's last tile also zero-fills up to
// the next boundary.  Thread i codes 4 consecutive keys (4 (i%32) ..) of 16
// channels (16 (i/32) ..) and packs each channel's 4 codes into one 32-bit
// word, so a warp stores 32 consecutive words of one channel row.
__global__ void __launch_bounds__(256) vquant_kernel(Fp8QuantArgs a) {
  constexpr int kRowWords = 36;  // 32 words of keys + 4 of padding (rows stay 16-byte aligned)
  __shared__ __align__(16) uint32_t tile[128 * kRowWords];
  __shared__ float rc[128];  // per-channel 448 / amax
  const int4 te = a.tiles[blockIdx.x];
  const int h = blockIdx.y;
  const int n = te.y - te.x;
  if (threadIdx.x < 128)
    rc[threadIdx.x] = fp8_recip(__uint_as_float(reinterpret_cast<const uint32_t*>(a.sv)[h * kHeadDim + threadIdx.x]));
  __syncthreads();
  const int tq = threadIdx.x & 31, cg = threadIdx.x >> 5;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.v) + (int64_t)te.x * a.stride + h * kHeadDim + cg * 16;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int ch0 = cg * 16 + half * 8;
    uint32_t pr[4][4];  // [key][channel pair]: two codes, the even channel's in the low byte
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * tq + i;
      float f[8];
      if (t < n) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(x + (int64_t)t * a.stride + half * 8)), f);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = 0.f;
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
        pr[i][p] = e4m3x2(__fmul_rn(f[2 * p], rc[ch0 + 2 * p]), __fmul_rn(f[2 * p + 1], rc[ch0 + 2 * p + 1]));
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t lo = pr[0][p] | (pr[1][p] << 16), hi = pr[2][p] | (pr[3][p] << 16);
      tile[(ch0 + 2 * p) * kRowWords + tq] = __byte_perm(lo, hi, 0x6420);      // even channel, keys 0..3
      tile[(ch0 + 2 * p + 1) * kRowWords + tq] = __byte_perm(lo, hi, 0x7531);  // odd channel
    }
  }
  __syncthreads();
  // thread i writes channel i/2, keys [64 (i%2), +64) as 16-byte pieces
  const int ch = threadIdx.x >> 1, k0 = (threadIdx.x & 1) * 64;
  const int n16 = (n + 15) / 16 * 16;
  uint8_t* out = static_cast<uint8_t*>(a.v8t) + ((int64_t)h * kHeadDim + ch) * a.v_pad + te.z + k0;
#pragma unroll
  for (int p = 0; p < 4; ++p)
    if (k0 + p * 16 < n16)
      *reinterpret_cast<uint4*>(out + p * 16) = *reinterpret_cast<const uint4*>(&tile[ch * kRowWords + k0 / 4 + 4 * p]);
}

__global__ void vscale_kernel(Fp8QuantArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < a.H * kHeadDim) a.sv[i] = fp8_scale(__uint_as_float(reinterpret_cast<const uint32_t*>(a.sv)[i]));
}

// v: codes (transposed) and scales, once sv holds the channel maxima' bits
cudaError_t launch_v_codes(const Fp8QuantArgs& a, cudaStream_t stream) {
  vquant_kernel<<<dim3(a.n_tiles, a.H), 256, 0, stream>>>(a);
  vscale_kernel<<<(a.H * kHeadDim + 255) / 256, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int num_sms, cudaStream_t stream) {
  if (a.S == 0) return cudaSuccess;
  const int64_t n_rows = a.S * a.H;
  const int64_t want = (n_rows + 15) / 16;
  const int grid_rows = (int)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  quant_rows_kernel<<<grid_rows, 256, 0, stream>>>(a);
  quant_ktiles_kernel<<<dim3(a.n_tiles, a.H), 256, 0, stream>>>(a);
  cudaError_t e = cudaMemsetAsync(a.sv, 0, (size_t)a.H * kHeadDim * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  vmax_kernel<<<dim3((unsigned)((a.H * 16 + 127) / 128), (unsigned)((a.S + kVmaxTokens - 1) / kVmaxTokens)), 128, 0,
                 stream>>>(a);
  return launch_v_codes(a, stream);
}

cudaError_t launch_prologue_fp8(const PrologueArgs& p, const Fp8QuantArgs& a, cudaStream_t stream) {
  if (a.S == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.sv, 0, (size_t)a.H * kHeadDim * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  prologue_quant_kernel<<<dim3(a.n_tiles, a.H), 256, 0, stream>>>(p, a);
  return launch_v_codes(a, stream);
}

}  // namespace h3
