// Packed varlen non-causal attention, warp-level mma.sync scaffold.
//
// A CTA of 8 warps takes a work unit (up to 256 query rows of one head inside
// one document) in two halves of 128 rows; each warp owns 16 query rows with
// Q, the running max/sum and the O accumulator in registers.  Keys and values
// stream through shared memory in 64-row tiles (cp.async, double-buffered),
// only over the unit's own document, so no cross-document tile is touched;
// the last tile masks keys past the document end.  Online softmax in the
// exp2 domain with the softmax scale folded into one multiply.
//
// Pages: vllm.cpp PR #26 "feat(minimax-h3)", PR description (per-document
// bidirectional attention over cu_seqlens, causal=false) and the
// warp-per-query-row commit (online-softmax recurrence with f32 accumulation,
// Q read once).
#include <cuda_bf16.h>

#include "device_common.cuh"

namespace h3 {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerPass = kWarps * 16;      // 128
constexpr int kKeyTile = 64;
constexpr int kPad = 136;                      // smem row pitch (elements): conflict-free ldmatrix
constexpr int kTileElems = kKeyTile * kPad;
constexpr size_t kSmemBytes = (size_t)4 * kTileElems * 2;  // K and V, double-buffered

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Copy one 64-row K and V tile (rows r0.., clipped at S with zero fill).
__device__ __forceinline__ void load_kv_tile(const __nv_bfloat16* k, const __nv_bfloat16* v,
                                             int64_t stride, int64_t S, int head, int64_t r0,
                                             uint32_t ks, uint32_t vs) {
#pragma unroll
  for (int i = 0; i < (kKeyTile * 16) / kThreads; ++i) {
    const int c = threadIdx.x + i * kThreads;  // 16-byte chunk id
    const int row = c >> 4, col = (c & 15) * 8;
    const int64_t gr = r0 + row;
    const bool ok = gr < S;
    const int64_t off = (ok ? gr : 0) * stride + (int64_t)head * kHeadDim + col;
    const uint32_t so = (uint32_t)(row * kPad + col) * 2;
    cp_async16(ks + so, k + off, ok ? 16 : 0);
    cp_async16(vs + so, v + off, ok ? 16 : 0);
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_fwd_mma_kernel(ForwardArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t s_base = dev::smem_u32(smem);
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(a.v);
  __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

#pragma unroll 1
  for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
    const WorkUnit wu = a.units[u];
#pragma unroll 1
    for (int half = 0; half < kUnitRows / kRowsPerPass; ++half) {
      const int32_t q0 = wu.q_row0 + half * kRowsPerPass;
      if (q0 >= wu.kv_end) break;
      const int64_t rA = q0 + warp * 16 + g, rB = rA + 8;
      // Q fragments (A operand, row-major 16x16 per k-step)
      uint32_t qa[8][4];
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const int c = kb * 16 + 2 * t;
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(qg + rA * a.qkv_stride + wu.head * kHeadDim + c);
        const uint32_t* pb = reinterpret_cast<const uint32_t*>(qg + rB * a.qkv_stride + wu.head * kHeadDim + c);
        const bool oka = rA < a.S, okb = rB < a.S;
        qa[kb][0] = oka ? pa[0] : 0u;
        qa[kb][1] = okb ? pb[0] : 0u;
        qa[kb][2] = oka ? pa[4] : 0u;
        qa[kb][3] = okb ? pb[4] : 0u;
      }
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      float o[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

      const int n_tiles = (wu.kv_end - wu.kv_begin + kKeyTile - 1) / kKeyTile;
      __syncthreads();  // previous users of the tile buffers are done
      load_kv_tile(kg, vg, a.qkv_stride, a.S, wu.head, wu.kv_begin, s_base, s_base + 2 * kTileElems * 2);
      cp_async_commit();
#pragma unroll 1
      for (int j = 0; j < n_tiles; ++j) {
        const int buf = j & 1;
        if (j + 1 < n_tiles) {
          const int nb = buf ^ 1;
          load_kv_tile(kg, vg, a.qkv_stride, a.S, wu.head, wu.kv_begin + (int64_t)(j + 1) * kKeyTile,
                       s_base + nb * kTileElems * 2, s_base + (2 + nb) * kTileElems * 2);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t ks = s_base + buf * kTileElems * 2;
        const uint32_t vs = s_base + (2 + buf) * kTileElems * 2;

        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
          for (int kb = 0; kb < 8; kb += 2) {
            const int mi = lane >> 3;
            const int row = nt * 8 + (lane & 7);
            const int col = (kb + (mi >> 1)) * 16 + (mi & 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ks + (uint32_t)(row * kPad + col) * 2, b0, b1, b2, b3);
            mma16816(s[nt], qa[kb], b0, b1);
            mma16816(s[nt], qa[kb + 1], b2, b3);
          }
        }
        // scale into the exp2 domain, mask keys past the document end
        const int key0 = wu.kv_begin + j * kKeyTile;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = key0 + nt * 8 + 2 * t + (e & 1);
            const float x = s[nt][e] * a.scale_log2;
            s[nt][e] = key < wu.kv_end ? x : -INFINITY;
          }
          mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
          mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = dev::ex2_approx(m0 - mn0), al1 = dev::ex2_approx(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const float p0 = dev::ex2_approx(s[nt][0] - mn0), p1 = dev::ex2_approx(s[nt][1] - mn0);
          const float p2 = dev::ex2_approx(s[nt][2] - mn1), p3 = dev::ex2_approx(s[nt][3] - mn1);
          rs0 += p0 + p1;
          rs1 += p2 + p3;
          pa[nt >> 1][(nt & 1) * 2 + 0] = dev::pack_bf16x2(p0, p1);
          pa[nt >> 1][(nt & 1) * 2 + 1] = dev::pack_bf16x2(p2, p3);
        }
        l0 = l0 * al0 + rs0;
        l1 = l1 * al1 + rs1;
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
          o[dn][0] *= al0;
          o[dn][1] *= al0;
          o[dn][2] *= al1;
          o[dn][3] *= al1;
        }
        // O += P V; P's A fragment for keys [16kb, 16kb+16) is (s tile 2kb, 2kb+1)
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint32_t af[4] = {pa[kb][0], pa[kb][1], pa[kb][2], pa[kb][3]};
#pragma unroll
          for (int dn = 0; dn < 16; dn += 2) {
            const int mi = lane >> 3;
            const int row = kb * 16 + (mi & 1) * 8 + (lane & 7);
            const int col = (dn + (mi >> 1)) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vs + (uint32_t)(row * kPad + col) * 2, b0, b1, b2, b3);
            mma16816(o[dn], af, b0, b1);
            mma16816(o[dn + 1], af, b2, b3);
          }
        }
        __syncthreads();  // all warps done with this buffer before it is refilled
      }
      cp_async_wait<0>();
      // epilogue
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
      }
      const float inv0 = 1.f / l0, inv1 = 1.f / l1;
      const bool okA = rA < wu.kv_end, okB = rB < wu.kv_end;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int c = dn * 8 + 2 * t;
        if (okA)
          *reinterpret_cast<uint32_t*>(og + rA * a.o_stride + wu.head * kHeadDim + c) =
              dev::pack_bf16x2(o[dn][0] * inv0, o[dn][1] * inv0);
        if (okB)
          *reinterpret_cast<uint32_t*>(og + rB * a.o_stride + wu.head * kHeadDim + c) =
              dev::pack_bf16x2(o[dn][2] * inv1, o[dn][3] * inv1);
      }
      if (a.lse != nullptr && t == 0) {
        const float ln2 = 0.6931471805599453f;
        if (okA) a.lse[(int64_t)wu.head * a.S + rA] = (m0 + __log2f(l0)) * ln2;
        if (okB) a.lse[(int64_t)wu.head * a.S + rB] = (m1 + __log2f(l1)) * ln2;
      }
    }
  }
}

}  // namespace

cudaError_t launch_forward_mma(const ForwardArgs& a, int num_sms, cudaStream_t stream,
                               std::string* why) {
  if (a.n_units == 0) return cudaSuccess;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) {
      if (why) *why = "cudaFuncSetAttribute failed";
      return e;
    }
    configured = true;
  }
  const int grid = a.n_units < num_sms ? a.n_units : num_sms;
  attn_fwd_mma_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace h3
