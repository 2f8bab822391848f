// Packed varlen non-causal attention on the 5th-generation tensor cores.
//
// Pages: vllm.cpp PR #26 "feat(minimax-h3)", PR description (packed varlen
// NON-CAUSAL attention: each query attends to every key of its own
// cu_seqlens document and to nothing else -- a cu_seqlens varlen
// flash-attention call with causal=false) and the warp-per-query-row commit
// (online-softmax recurrence in f32; Q read once per query row).
//
// Design (one persistent CTA per SM, 10 warps):
//   warp 9       TMA producer: Q tiles of the work unit, then the unit's
//                document's K and V tiles through a 4-slot shared-memory ring,
//                V(j) and the next K tile loaded as one group behind one
//                barrier (one readiness poll and one release per key tile).
//   warp 8       MMA issuer (one thread) and TMEM owner: S_s = Q_s K_j^T and
//                O_s += P_s V_j with tcgen05.mma, fp32 accumulators in TMEM.
//   warps 0..3   softmax for query tile 0 (rows 0..127 of the unit),
//   warps 4..7   softmax for query tile 1 (rows 128..255): one thread per
//                query row reads its S row from TMEM, keeps the running max
//                and sum in registers (no cross-thread reduction is needed
//                since a thread owns a whole row), writes P as bf16 back into
//                TMEM over its S columns, rescales its O row when the max has
//                grown by more than 2^8, and at the end of the unit writes
//                O / l and the log-sum-exp.
// While one softmax group works on its tile, the tensor core runs the other
// tile's MMAs (two-tile ping-pong).  A work unit (head, document, 256 query
// rows) only visits its own document's key tiles; keys past the document end
// in the last tile are masked to -inf, rows past it are never stored.
//
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512); P_s is
// bf16 packed two per column in the first 64 columns of S_s.
//
// Shared memory tiles are 128 rows x 64 bf16 (128 B per row, 128-byte TMA
// swizzle); a 128 x 128 tile is two of them 16 KB apart.  Q and K are K-major
// operands; V is the MN-major B operand of the PV product.
//
// Every mbarrier wait is bounded (mbar_wait_bounded): on expiry the CTA
// raises an abort flag, records a timeout in the device error word, drains
// its own copies and MMAs with bounded waits, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"

namespace h3 {

namespace {

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kTileRows = 128;
constexpr int kSlots = 4;
constexpr uint32_t kHalfTileBytes = 128 * 128;        // 128 rows x 128 B
constexpr uint32_t kTileBytes = 2 * kHalfTileBytes;   // 32 KB
constexpr uint32_t kSmemQ = 0;                        // 2 tiles
constexpr uint32_t kSmemKV = 2 * kTileBytes;          // kSlots tiles
constexpr uint32_t kSmemBar = kSmemKV + kSlots * kTileBytes;
// barriers: q_full[2] q_empty[2] kv_full[4] kv_empty[4] s_ready[2] p_ready[2] o_ready[2] drain
constexpr int kNumBars = 2 + 2 + kSlots + kSlots + 2 + 2 + 2 + 1;
constexpr uint32_t kSmemMisc = kSmemBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kSmemMisc + 16;
constexpr size_t kSmemAlloc = kSmemBytes + 1024;      // slack to align the base to 1 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;        // 2 s
constexpr float kRescaleThreshold = 8.0f;             // log2 units: rescale when max grows by > 2^8

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, M = 128, N = 128.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBase;             // A, B K-major
constexpr uint32_t kIdescPV = kIdescBase | (1u << 16);  // B (V) MN-major

// Shared-memory matrix descriptor with 128-byte swizzling.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

struct Bars {
  uint32_t base;
  __device__ uint32_t q_full(int s) const { return base + 8 * s; }
  __device__ uint32_t q_empty(int s) const { return base + 8 * (2 + s); }
  __device__ uint32_t kv_full(int i) const { return base + 8 * (4 + i); }
  __device__ uint32_t kv_empty(int i) const { return base + 8 * (4 + kSlots + i); }
  __device__ uint32_t s_ready(int s) const { return base + 8 * (4 + 2 * kSlots + s); }
  __device__ uint32_t p_ready(int s) const { return base + 8 * (6 + 2 * kSlots + s); }
  __device__ uint32_t o_ready(int s) const { return base + 8 * (8 + 2 * kSlots + s); }
  __device__ uint32_t drain() const { return base + 8 * (10 + 2 * kSlots); }
};

struct UnitGeom {
  int32_t q0, kv0, kv1, head, lo, hi, part, n_st;  // key tiles [lo, hi)
};

__device__ __forceinline__ UnitGeom unit_geom(const WorkUnit* units, int u) {
  const int4 w = __ldg(reinterpret_cast<const int4*>(units) + 2 * u);
  const int4 x = __ldg(reinterpret_cast<const int4*>(units) + 2 * u + 1);
  UnitGeom g;
  g.q0 = w.x;
  g.kv0 = w.y;
  g.kv1 = w.z;
  g.head = w.w;
  g.lo = x.x;
  g.hi = x.y;
  g.part = x.z;
  g.n_st = (w.x + kTileRows < w.z) ? 2 : 1;
  return g;
}

// One 128-row tile of K or V (two 64-column boxes) into a ring slot.
__device__ __forceinline__ void load_kv_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int head,
                                             int32_t row, uint64_t pol) {
  dev::tma_load_2d(dst, tm, bar, head * 128, row, pol);
  dev::tma_load_2d(dst + kHalfTileBytes, tm, bar, head * 128 + 64, row, pol);
}

// S (TMEM, 128 x 128 fp32) = Q (smem, K-major) * K^T (smem, K-major), 8 MMAs of K = 16.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfTileBytes + (kk & 3) * 32;
    dev::mma_ss(d_tmem, smem_desc(q_smem + off, 16, 1024), smem_desc(k_smem + off, 16, 1024), kIdescQK,
                kk > 0 ? 1u : 0u);
  }
}

// O (TMEM fp32) (+)= P (TMEM, bf16 pairs) * V (smem, MN-major), 8 MMAs of K = 16 keys.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    dev::mma_ts(d_tmem, p_tmem + kk * 8, smem_desc(v_smem + kk * 16 * 128, kHalfTileBytes, 1024), kIdescPV,
                (acc || kk > 0) ? 1u : 0u);
}

// One query row's 128 scores from TMEM (4 loads of 32 columns); keys past
// the document end (column >= rem) are set to -inf.
__device__ __forceinline__ void load_scores(uint32_t t_s, uint32_t (&r)[4][32], int rem) {
#pragma unroll
  for (int c = 0; c < 4; ++c) dev::tmem_ld32(t_s + c * 32, r[c]);
  dev::tmem_wait_ld();
  if (rem < kTileRows) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= rem) r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, ForwardArgs a) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  const Bars bars{sbase + kSmemBar};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  const uint32_t warp = dev::warp_id_uniform();
  const uint32_t lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      dev::mbar_init(bars.q_full(s), 1);
      dev::mbar_init(bars.q_empty(s), 1);
      dev::mbar_init(bars.s_ready(s), 1);
      dev::mbar_init(bars.p_ready(s), kTileRows);
      dev::mbar_init(bars.o_ready(s), 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      dev::mbar_init(bars.kv_full(i), 1);
      dev::mbar_init(bars.kv_empty(i), 1);
    }
    dev::mbar_init(bars.drain(), 1);
    dev::fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    dev::tma_prefetch_desc(&tm_q);
    dev::tma_prefetch_desc(&tm_k);
    dev::tma_prefetch_desc(&tm_v);
  }
  if (warp == kMmaWarp) {
    dev::tmem_alloc(dev::smem_u32(tmem_slot), kTmemCols);
    dev::tmem_relinquish();
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------ TMA producer ----
    if (lane == 0) {
      const uint64_t pol_q = dev::policy_evict_first();
      const uint64_t pol_kv = dev::policy_evict_last();
      uint32_t grp = 0, q_it[2] = {0, 0};
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
        const UnitGeom g = unit_geom(a.units, u);
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!ok || s >= g.n_st) break;
          ok = dev::mbar_wait(bars.q_empty(s), (q_it[s] & 1) ^ 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          const uint32_t dst = sbase + kSmemQ + s * kTileBytes;
          dev::mbar_arrive_expect_tx(bars.q_full(s), kTileBytes);
          const int32_t row = g.q0 + s * kTileRows;
          dev::tma_load_2d(dst, &tm_q, bars.q_full(s), g.head * 128, row, pol_q);
          dev::tma_load_2d(dst + kHalfTileBytes, &tm_q, bars.q_full(s), g.head * 128 + 64, row, pol_q);
          ++q_it[s];
        }
        // Key/value groups: group 0 is the first unit's first K tile (ring slot
        // 0); group n >= 1 is V(j) with the next K tile -- K(j+1), or the next
        // unit's first K tile -- in slots (2n-1) % 4 and 2n % 4, one full and
        // one empty barrier (index n & 1) for both.
        if (u == (int)blockIdx.x) {
          ok = dev::mbar_wait(bars.kv_empty(0), 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          dev::mbar_arrive_expect_tx(bars.kv_full(0), kTileBytes);
          load_kv_tile(sbase + kSmemKV, &tm_k, bars.kv_full(0), g.head, g.kv0 + g.lo * kTileRows, pol_kv);
          grp = 1;
        }
        for (int j = g.lo; ok && j < g.hi; ++j) {
          bool has_k = j + 1 < g.hi;
          int k_head = g.head;
          int32_t k_row = g.kv0 + (j + 1) * kTileRows;
          if (!has_k && u + (int)gridDim.x < a.n_units) {
            const UnitGeom n = unit_geom(a.units, u + gridDim.x);
            has_k = true;
            k_head = n.head;
            k_row = n.kv0 + n.lo * kTileRows;
          }
          const uint32_t b = grp & 1;
          ok = dev::mbar_wait(bars.kv_empty(b), ((grp >> 1) & 1) ^ 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          dev::mbar_arrive_expect_tx(bars.kv_full(b), has_k ? 2 * kTileBytes : kTileBytes);
          load_kv_tile(sbase + kSmemKV + ((2 * grp - 1) % kSlots) * kTileBytes, &tm_v, bars.kv_full(b), g.head,
                       g.kv0 + j * kTileRows, pol_kv);
          if (has_k)
            load_kv_tile(sbase + kSmemKV + ((2 * grp) % kSlots) * kTileBytes, &tm_k, bars.kv_full(b), k_head, k_row,
                         pol_kv);
          ++grp;
        }
      }
      if (!ok) {
        // drain: wait (bounded) for every copy this thread issued into the ring and Q
        for (uint32_t r = 1; r <= 2 && r <= grp; ++r) {
          const uint32_t n = grp - r;
          dev::mbar_wait_bounded(bars.kv_full(n & 1), (n >> 1) & 1, nullptr, nullptr, kTimeoutNs);
        }
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (q_it[s]) dev::mbar_wait_bounded(bars.q_full(s), (q_it[s] - 1) & 1, nullptr, nullptr, kTimeoutNs);
      }
    }
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------- MMA issuer ----
    if (lane == 0) {
      uint32_t grp = 0, q_it0 = 0, q_it1 = 0, p_it0 = 0, p_it1 = 0;
      bool ok = true;
      bool issued = false;
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
        const UnitGeom g = unit_geom(a.units, u);
        const bool last_unit = u + (int)gridDim.x >= a.n_units;
        ok = dev::mbar_wait(bars.q_full(0), q_it0 & 1, abort_flag, a.err, kTimeoutNs);
        ++q_it0;
        if (ok && g.n_st > 1) {
          ok = dev::mbar_wait(bars.q_full(1), q_it1 & 1, abort_flag, a.err, kTimeoutNs);
          ++q_it1;
        }
        // this unit's first K tile: group 0 (first unit) or the K half of the
        // previous unit's last group (already waited for)
        uint32_t k0, rel;
        if (u == (int)blockIdx.x) {
          if (ok) ok = dev::mbar_wait(bars.kv_full(0), 0, abort_flag, a.err, kTimeoutNs);
          k0 = 0;
          rel = 0;
          grp = 1;
        } else {
          k0 = (2 * (grp - 1)) % kSlots;
          rel = grp - 1;
        }
        if (!ok) break;
        dev::tc_fence_after();
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (s >= g.n_st) break;
          issue_qk(tmem + s * 128, sbase + kSmemQ + s * kTileBytes, sbase + kSmemKV + k0 * kTileBytes);
          dev::mma_commit(bars.s_ready(s));
          if (g.hi - g.lo == 1) dev::mma_commit(bars.q_empty(s));
        }
        dev::mma_commit(bars.kv_empty(rel & 1));  // that K tile (and the V tile before it) are done
        issued = true;
        for (int j = g.lo; j < g.hi; ++j) {
          const uint32_t b = grp & 1;
          const uint32_t vslot = (2 * grp - 1) % kSlots, kslot = (2 * grp) % kSlots;
          const bool more = j + 1 < g.hi;
          ok = dev::mbar_wait(bars.kv_full(b), (grp >> 1) & 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (s >= g.n_st) break;
            uint32_t& p_it = s == 0 ? p_it0 : p_it1;
            ok = dev::mbar_wait(bars.p_ready(s), p_it & 1, abort_flag, a.err, kTimeoutNs);
            if (!ok) break;
            ++p_it;
            dev::tc_fence_after();
            issue_pv(tmem + 256 + s * 128, tmem + s * 128, sbase + kSmemKV + vslot * kTileBytes, j > g.lo);
            if (more) {
              issue_qk(tmem + s * 128, sbase + kSmemQ + s * kTileBytes, sbase + kSmemKV + kslot * kTileBytes);
              dev::mma_commit(bars.s_ready(s));
              if (j + 2 == g.hi) dev::mma_commit(bars.q_empty(s));
            } else {
              dev::mma_commit(bars.o_ready(s));
            }
          }
          if (!ok) break;
          // V(j) and K(j+1) are done; a unit's last group also holds the next
          // unit's first K tile and is released after that QK (next prologue)
          if (more || last_unit) dev::mma_commit(bars.kv_empty(b));
          ++grp;
        }
      }
      if (!ok && issued) {
        // drain: every MMA issued so far must finish before TMEM is freed
        dev::mma_commit(bars.drain());
        dev::mbar_wait_bounded(bars.drain(), 0, nullptr, nullptr, kTimeoutNs);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax ----
    const int st = warp >> 2;            // query tile of this warpgroup
    const uint32_t row_in_tile = threadIdx.x & 127;
    const uint32_t lane_base = (warp & 3) * 32;
    const uint32_t t_s = tmem + (lane_base << 16) + st * 128;        // S_s / P_s
    const uint32_t t_o = tmem + (lane_base << 16) + 256 + st * 128;  // O_s
    uint32_t s_it = 0, o_it = 0;
    bool ok = true;
    const float sl2 = a.scale_log2;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const UnitGeom g = unit_geom(a.units, u);
      if (st >= g.n_st) continue;
      float m_used = -INFINITY, l = 0.f;
      for (int j = g.lo; j < g.hi; ++j) {
        ok = dev::mbar_wait(bars.s_ready(st), s_it & 1, abort_flag, a.err, kTimeoutNs);
        if (!ok) break;
        ++s_it;
        __syncwarp();  // lanes leave the wait separately; the TMEM loads are warp-collective
        dev::tc_fence_after();
        uint32_t r[4][32];
        float* sv = reinterpret_cast<float*>(&r[0][0]);
        const int rem = g.kv1 - (g.kv0 + j * kTileRows);
        load_scores(t_s, r, rem);
        // Row max: eight independent chains of 3-input maxima.
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = dev::max3(mx[i], sv[c + i], sv[c + 8 + i]);
        const float m_new =
            dev::max3(dev::max3(mx[0], mx[1], mx[2]), dev::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
        // The reference max only moves when the row max grows by more than
        // 2^8 (then O and l are rescaled; the final O / l is unchanged).  The
        // O row is rescaled after P is written: the next PV waits for p_ready.
        float alpha = 1.f;
        if (m_new > m_used + kRescaleThreshold) {
          alpha = dev::ex2_approx(m_used - m_new);  // 0 on the first tile (m_used = -inf)
          m_used = m_new;
        }
        const float neg = -m_used;
        float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t p[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            // packed pair arithmetic: one f32x2 FMA for the exponents, one f32x2 add for the sums
            float x0, x1;
            dev::fma2(x0, x1, sv[64 * h + 2 * c], sv[64 * h + 2 * c + 1], sl2, sl2, neg, neg);
            const float p0 = dev::ex2_approx(x0), p1 = dev::ex2_approx(x1);
            const int ai = 2 * (c & 3);
            dev::add2(rs8[ai], rs8[ai + 1], rs8[ai], rs8[ai + 1], p0, p1);
            p[c] = dev::pack_bf16x2(p0, p1);
          }
          dev::tmem_st32(t_s + 32 * h, p);
        }
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        l = l * alpha + rs;
        // tcgen05.ld/st are warp-collective (.sync.aligned): the rescale runs
        // for the whole warp when any of its rows needs it (alpha = 1 elsewhere).
        if (j > g.lo && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            dev::tmem_ld32(t_o + c * 32, ov);
            dev::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            dev::tmem_st32(t_o + c * 32, ov);
          }
        }
        dev::tmem_wait_st();
        dev::tc_fence_before();
        dev::mbar_arrive(bars.p_ready(st));
      }
      if (!ok) break;
      ok = dev::mbar_wait(bars.o_ready(st), o_it & 1, abort_flag, a.err, kTimeoutNs);
      if (!ok) break;
      ++o_it;
      __syncwarp();
      dev::tc_fence_after();
      const int32_t row = g.q0 + st * kTileRows + row_in_tile;
      const bool valid = row < g.kv1;
      if (g.part >= 0) {
        // A piece of a unit split along the keys: unnormalised O row, its
        // reference max (log2 units) and sum, for the merge pass.
        const size_t slot = (size_t)g.part * kUnitRows + st * kTileRows + row_in_tile;
        float4* dst = reinterpret_cast<float4*>(a.part_o + slot * kHeadDim);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          dev::tmem_ld32(t_o + c * 32, ov);
          dev::tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[c * 8 + e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                           __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
          }
        }
        if (valid) a.part_ml[slot] = make_float2(m_used, l);
        continue;
      }
      const float inv = 1.f / l;
      __nv_bfloat16* dst = og + (int64_t)row * a.o_stride + g.head * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        dev::tmem_ld32(t_o + c * 32, ov);
        dev::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = dev::pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
            w.y = dev::pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
            w.z = dev::pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
            w.w = dev::pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + e * 8) = w;
          }
        }
      }
      if (valid && a.lse != nullptr)
        a.lse[(int64_t)g.head * a.S + row] = (m_used + __log2f(l)) * 0.6931471805599453f;
    }
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();  // lane 0 comes from the issue loop; dealloc is warp-collective
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, kTmemCols);
  }
}

// Combines the pieces of units split along the keys: one warp per query row,
// four dims per lane.  With M = max_c m_c (log2 units):
//   o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  lse = (M + log2 l) ln 2.
__global__ void __launch_bounds__(256) attn_merge_kernel(ForwardArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int mu = warp_global / kUnitRows, r = warp_global % kUnitRows;
  if (mu >= a.n_merges) return;
  const MergeUnit m = a.merges[mu];
  const int32_t row = m.q_row0 + r;
  if (row >= m.kv_end) return;
  float M = -INFINITY;
  for (int c = 0; c < m.n_parts; ++c) M = fmaxf(M, a.part_ml[(size_t)(m.part0 + c) * kUnitRows + r].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int c = 0; c < m.n_parts; ++c) {
    const size_t slot = (size_t)(m.part0 + c) * kUnitRows + r;
    const float2 ml = a.part_ml[slot];
    const float w = dev::ex2_approx(ml.x - M);
    const float4 o = reinterpret_cast<const float4*>(a.part_o + slot * kHeadDim)[lane];
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
    l = fmaf(w, ml.y, l);
  }
  const float inv = 1.f / l;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.o) + (int64_t)row * a.o_stride + m.head * kHeadDim + 4 * lane;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(dev::pack_bf16x2(acc.x * inv, acc.y * inv), dev::pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0 && a.lse != nullptr) a.lse[(int64_t)m.head * a.S + row] = (M + __log2f(l)) * 0.6931471805599453f;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int64_t S, int32_t H, int64_t stride, std::string* why) {
  auto fn = encode_fn();
  if (fn == nullptr) {
    if (why) *why = "cuTensorMapEncodeTiled is unavailable";
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)H * kHeadDim, (cuuint64_t)S};
  cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  cuuint32_t box[2] = {64, kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

}  // namespace

cudaError_t launch_forward(const ForwardArgs& a, int num_sms, cudaStream_t stream, std::string* why) {
  if (a.n_units == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.S, a.H, a.qkv_stride, why) || !make_map(&mk, a.k, a.S, a.H, a.qkv_stride, why) ||
      !make_map(&mv, a.v, a.S, a.H, a.qkv_stride, why))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  });
  if (attr != cudaSuccess) {
    if (why) *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return attr;
  }
  const int grid = a.n_units < num_sms ? a.n_units : num_sms;
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.n_merges == 0) return e;
  const int64_t warps = (int64_t)a.n_merges * kUnitRows;
  attn_merge_kernel<<<(int)((warps + 7) / 8), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace h3
