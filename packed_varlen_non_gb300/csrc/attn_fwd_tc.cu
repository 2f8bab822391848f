// Packed varlen non-causal attention on the 5th-generation tensor cores,
// run by CTA pairs.
//
// Pages: vllm.cpp PR #26 "feat(minimax-h3)", PR description (packed varlen
// NON-CAUSAL attention: each query attends to every key of its own
// cu_seqlens document and to nothing else -- a cu_seqlens varlen
// flash-attention call with causal=false) and the warp-per-query-row commit
// (online-softmax recurrence in f32; Q read once per query row).
//
// Design: a cluster of two CTAs (one per SM of a pair) works on one unit of
// 512 query rows of one (head, document); each CTA owns 256 of them as two
// 128-row query tiles s = 0, 1 (rows q0 + 256 s + 128 rank + i).  The MMAs are
// pair instructions (tcgen05 cta_group::2, M = 256): one thread of the even
// CTA issues them, each CTA's tensor core computes its own 128 rows, and each
// CTA holds only half of every B operand -- keys [64 rank, 64 rank + 64) of a
// K tile and dims [64 rank, 64 rank + 64) of a V tile -- so a CTA reads
// (and loads from L2) half the key/value bytes a single-CTA kernel would.
// Per CTA, 11 warps:
//   warp 9       lane 0: TMA producer, its halves of the document's K and V
//                tiles through a 6-slot ring; V(j) and the next K tile form
//                one group behind one barrier.  (FP8: also its own Q tiles,
//                the next unit's behind the current unit's first K/V group.)
//                lane 1 (bf16): the O-store thread (below).
//   warp 10      Q warp: loads this CTA's Q tiles (bf16) into double-buffered
//                slots as they come free, so the next unit's tiles are ready
//                before it starts; as each lands, applies the fused Q prologue
//                in place when asked (RMSNorm with gain, rot96 rotation) and
//                reports the tile ready to the even CTA.
//   warp 8       even CTA: MMA issuer for the pair, S = Q_s K^T and
//                O_s += P V, fp32 accumulators in TMEM.  Both CTAs' warp 8
//                allocate the pair's TMEM together.
//   warps 0..3   softmax for query tile 0 of this CTA,
//   warps 4..7   softmax for query tile 1: one thread per query row reads its
//                S row from TMEM, keeps the running max and sum in registers,
//                writes P as bf16 back into TMEM over its S columns, rescales
//                its O row when the max has grown by more than 2^8, and at the
//                end of the unit writes O / l and the log-sum-exp.  A bf16
//                warp whose 32 rows all lie in the document stages them, bf16,
//                in the unit's Q slot (free once the unit's MMAs are done);
//                other warps store their rows directly.  Either way the four
//                warps of a query tile then report to the O-store thread,
//                which sends the staged rows out with TMA tile stores, waits
//                until they have read the slot and frees it for the Q warp --
//                so the softmax warps never wait on the TMA unit.
// Each 128-key tile is taken in two halves of 64 keys, h = 0, 1, each with
// its own 64 TMEM columns of S: per query tile the issuer runs PV of half h
// of key tile j and then QK of half h of key tile j + 1 into the same
// columns, so the softmax works on the other half while the tensor cores
// compute the next S half -- a query tile's softmax does not wait for its own
// PV and next QK.  Both query tiles and both halves interleave on the tensor
// pipe (order per key tile: tile 0 half 0, tile 1 half 0, tile 0 half 1,
// tile 1 half 1).  A unit only visits its own document's key tiles; keys past
// the document end in the last tile are masked to -inf, rows past it are
// never stored.  Each pair runs its own range of the work list (placed on the
// host longest-processing-time first), and the next unit's first QKs are
// issued right after the current unit's last PVs, so its softmax finds them
// done when it comes back from the epilogue.
//
// Key halves: a CTA holds keys [64 rank, 64 rank + 64) of a tile; half h is
// rows [32 h, 32 h + 32) of both CTAs' halves (the pair MMA takes B's first
// 32 columns from the even CTA), so S column c of half h is key 32 h + c for
// c < 32 and 64 + 32 h + (c - 32) for c >= 32; the PV of a half reads the
// matching 16-key (bf16) or 32-key (FP8) chunks of V.
//
// TMEM columns (each CTA): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512),
// S_s half h at S_s + 64 h; P of a half is bf16 packed two per column in the
// half's first 32 columns.
//
// Shared memory rows are 64 bf16 (128 B, 128-byte TMA swizzle).  Q tiles are
// 128 rows x 128 dims (two 16 KB halves); a K half-tile is 64 keys x 128 dims
// (two 8 KB halves), a V half-tile 128 keys x 64 dims (16 KB).  Q and K are
// K-major operands; V is the MN-major B operand of the PV product.
//
// Barriers: completion of the pair's MMAs is multicast to both CTAs (S half
// ready, PV done; FP8: Q slots free).  The MMA-issuing thread paces the tensor
// cores, so per key-tile half it only waits for P and commits: its "P ready"
// barrier of (query tile, half) counts one arrival per softmax warp of both
// CTAs, and softmax warp 0 of each CTA reports half 0 only once its CTA's next
// K/V group has landed; a softmax thread of the unit's last query tile that
// sees S half 1 of key tile t ready frees the ring slots of the group holding
// K(t) (everything before that QK has completed).  "PV done" of a query tile
// and half completes once per unit, after the PV of that half in the unit's
// last key tile: the epilogue waits for both halves.  A rescale of O first
// waits for the other half's latest PV: through the S-ready of the QK issued
// right after it, or "PV done" in the last key tile.  Q tiles:
// the even CTA's "Q ready" barrier counts one arrival from the Q warp of each
// CTA; a bf16 Q slot is freed by the O-store thread after the four softmax
// warps of its query tile in that CTA have reported their epilogue done.
//
// FP8 variant (template argument kFp8, h3attn_forward_fp8): the same kernel
// on e4m3 Q, K and transposed V (channel rows of keys, every document
// starting on a 16-key boundary) with fp32 scales -- kind::f8f6f4 pair MMAs of
// K = 32, 16 KB Q tiles and 8 KB half-tiles in 128-byte rows, P rounded to
// e4m3 and stored four per TMEM column (first 32 columns of S), the q-row x
// key-tile scale folded into the softmax's score multiplier, the per-channel
// V scale applied to O in the epilogue.  Its MMAs are half as long as bf16's,
// so it keeps whole 128-key tiles (one S-ready and one P-ready phase per key
// tile and query tile, P over S, issued by one thread): split into halves,
// the per-half softmax costs measured slower than the chain they remove.
//
// Every mbarrier wait is bounded: on expiry the CTA raises an abort flag,
// records a timeout in the device error word, drains its own copies and MMAs
// with bounded waits, and leaves through the cluster barrier, where the pair
// frees its TMEM together.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "device_common.cuh"
#include "qk_norm.cuh"

namespace h3 {

namespace {

constexpr int kThreads = 352;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kQWarp = 10;
constexpr int kTileRows = 128;
constexpr int kSlots = 6;                              // ring slots (16 KB each)
constexpr int kGroups = kSlots / 2;                    // key/value groups in flight
// barriers: q_full[4] q_empty[4] q_ready[4] kv_full[G] kv_empty[G] s_ready[2][2] p_ready[2][2] pv_done[2][2] drain o_staged[4]
constexpr int kNumBars = 12 + 2 * kGroups + 4 + 4 + 4 + 1 + 4;
// Shared-memory layout: 2 buffers x 2 query tiles, then the ring.  bf16: a Q
// tile is 128 rows x 128 dims in two 16 KB halves of 64 dims, a slot 16 KB;
// fp8 (e4m3): a Q tile is one 16 KB block of 128-byte rows, a slot 8 KB.
template <bool kFp8>
struct Cfg {
  static constexpr uint32_t QTileBytes = kFp8 ? 128 * 128 : 128 * 128 * 2;
  static constexpr uint32_t SlotBytes = kFp8 ? 64 * 128 : 64 * 128 * 2;
  static constexpr uint32_t SmemQ = 0;
  static constexpr uint32_t SmemKV = 4 * QTileBytes;
  static constexpr uint32_t SmemBar = SmemKV + kSlots * SlotBytes;
  static constexpr uint32_t SmemMisc = SmemBar + kNumBars * 8;
  static constexpr size_t SmemAlloc = SmemMisc + 16 + 1024;  // slack to align the base to 1 KB
  static_assert(SmemAlloc <= 227 * 1024, "shared memory per CTA");
};
constexpr uint32_t kQHalfBytes = 128 * 128;            // bf16 Q tile: one half (64 dims)
constexpr uint32_t kKHalfBytes = 64 * 128;             // bf16 K half-tile: one half (64 dims)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;         // 2 s
constexpr float kRescaleThreshold = 8.0f;              // log2 units: rescale when max grows by > 2^8
constexpr uint16_t kPairMask = 0x3;
static_assert(kUnitRows == 4 * kTileRows, "a unit is two query tiles in each CTA of the pair");

// Instruction descriptors, kind::f16: fp32 accumulator, bf16 A and B, M = 256 (pair).
// QK: N = 64 keys (one half of a key tile), A and B K-major; PV: N = 128 dims,
// B (V) MN-major.
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((256u >> 4) << 24);
constexpr uint32_t kIdescQK = kIdescBf16 | ((64u >> 3) << 17);
constexpr uint32_t kIdescPV = kIdescBf16 | ((128u >> 3) << 17) | (1u << 16);
// kind::f8f6f4: e4m3 A and B (type code 0), fp32 accumulator, M = 256, N = 128,
// both K-major (the FP8 pipeline takes whole 128-key tiles)
constexpr uint32_t kIdescF8 = (1u << 4) | ((128u >> 3) << 17) | ((256u >> 4) << 24);

// Q slot i = 2 * buffer + query tile; the unit with ordinal k (per pair) uses buffer k & 1.
struct Bars {
  uint32_t base;
  __device__ uint32_t q_full(int i) const { return base + 8 * i; }
  __device__ uint32_t q_empty(int i) const { return base + 8 * (4 + i); }
  __device__ uint32_t q_ready(int i) const { return base + 8 * (8 + i); }
  __device__ uint32_t kv_full(int i) const { return base + 8 * (12 + i); }
  __device__ uint32_t kv_empty(int i) const { return base + 8 * (12 + kGroups + i); }
  // S of key-tile half h of query tile s is in TMEM / P of it is in TMEM
  __device__ uint32_t s_ready(int s, int h) const { return base + 8 * (12 + 2 * kGroups + 2 * s + h); }
  __device__ uint32_t p_ready(int s, int h) const { return base + 8 * (16 + 2 * kGroups + 2 * s + h); }
  // the PV of half h of query tile s in a unit's last key tile has completed
  // (one phase per unit)
  __device__ uint32_t pv_done(int s, int h) const { return base + 8 * (20 + 2 * kGroups + 2 * s + h); }
  __device__ uint32_t drain() const { return base + 8 * (24 + 2 * kGroups); }
  // bf16: the four softmax warps of Q slot i's query tile have finished that
  // unit's epilogue (their O rows staged in the slot or stored)
  __device__ uint32_t o_staged(int i) const { return base + 8 * (25 + 2 * kGroups + i); }
};

struct UnitGeom {
  int32_t q0, kv0, kv1, head, lo, hi, part, n_st;  // key tiles [lo, hi)
  int32_t v_off;                                   // FP8: the document's first key in the transposed V
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
  g.v_off = x.w;
  g.n_st = (w.x + 2 * kTileRows < w.z) ? 2 : 1;  // query tile 1 of the pair holds rows from 256 on
  return g;
}

// This CTA's half of a K tile: keys [key0 + 64 rank, +64), all 128 dims (bf16:
// two boxes of 64 dims; fp8: one box of 128-byte rows).
template <bool kFp8>
__device__ __forceinline__ void load_k_half(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int head,
                                            int32_t key0, uint32_t rank, uint64_t pol) {
  const int32_t row = key0 + 64 * (int32_t)rank;
  dev::tma_load_2d(dst, tm, bar, head * 128, row, pol);
  if constexpr (!kFp8) dev::tma_load_2d(dst + kKHalfBytes, tm, bar, head * 128 + 64, row, pol);
}

// This CTA's half of a V tile: 128 keys, dims [64 rank, 64 rank + 64) (one box;
// fp8: rows of the transposed V, one per channel, 128 keys each).
// key0: the tile's first key row (bf16) or its first key in the transposed V,
// a multiple of 16 (fp8).
template <bool kFp8>
__device__ __forceinline__ void load_v_half(uint32_t dst, const CUtensorMap* tm, uint32_t bar, int head,
                                            int32_t key0, uint32_t rank, uint64_t pol) {
  if constexpr (kFp8)
    dev::tma_load_2d(dst, tm, bar, key0, head * 128 + 64 * (int32_t)rank, pol);
  else
    dev::tma_load_2d(dst, tm, bar, head * 128 + 64 * (int32_t)rank, key0, pol);
}

// Shared-memory descriptors, split into 32-bit words: the high word (stride
// 1024 B between 8-row groups, descriptor version 1, 128-byte swizzle) is the
// same for every operand here; the low word holds the start address >> 4 and
// the leading-byte offset >> 4, and stepping through an operand only adds to
// the address field (addresses stay below 256 KB, so it never carries).
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t addr, uint32_t lbo) {
  return ((addr >> 4) & 0x3FFFu) | ((lbo >> 4) << 16);
}

// Key-tile halves.  Each CTA holds keys [64 rank, 64 rank + 64) of a 128-key
// tile; half h of the tile is rows [32 h, 32 h + 32) of both CTAs' halves (the
// pair MMA takes B's first 32 columns from the even CTA, the next 32 from the
// odd one), so S column c of half h is key 32 h + c (c < 32) or
// 64 + 32 h + (c - 32) (c >= 32) of the tile.  The half's 32 rows start
// 32 x 128 B = 4 KB into each CTA's K half-tile (a whole number of 1 KB swizzle
// atoms).
constexpr uint32_t kHalfKeyRowsBytes = 32 * 128;

// Key offset within the 128-key tile of S column c (0..63) of half h.
__device__ __forceinline__ int half_key(int c, int h) { return 32 * h + c + (c >= 32 ? 32 : 0); }

// S half (TMEM, 128 x 64 fp32 in each CTA) = Q (smem, K-major) * K^T (smem,
// K-major, 32 keys per CTA): 8 pair MMAs of K = 16 in one block.  Step kk
// reads Q at +(kk/4) 16 KB + (kk%4) 32 B and K at +(kk/4) 8 KB + (kk%4) 32 B.
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  const uint32_t qa = desc_lo(q_smem, 16), kb = desc_lo(k_smem, 16);
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 a, b;\n\t.reg .b32 x, y;\n\t"
      "setp.ne.u32 p0, %4, %4;\n\t"
      "setp.eq.u32 p1, %4, %4;\n\t"
      "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p0;\n\t"
      "add.u32 x, %1, 2;\n\tadd.u32 y, %2, 2;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 4;\n\tadd.u32 y, %2, 4;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 6;\n\tadd.u32 y, %2, 6;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 1024;\n\tadd.u32 y, %2, 512;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 1026;\n\tadd.u32 y, %2, 514;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 1028;\n\tadd.u32 y, %2, 516;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 1030;\n\tadd.u32 y, %2, 518;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a, b, %5, p1;\n\t}" ::"r"(d_tmem),
      "r"(qa), "r"(kb), "r"(kDescHi), "r"(0u), "r"(kIdescQK)
      : "memory");
}

// O (TMEM fp32) (+)= P (TMEM, bf16 pairs: 32 columns for the half's 64 keys)
// * V (smem, MN-major, 64 dims per CTA), 4 pair MMAs of K = 16 keys.  MMA i
// reads P columns +8 i, i.e. S columns [16 i, 16 i + 16) of the half, whose
// keys are V's 16-key chunk 2h + {0, 1, 4, 5}[i] (2 KB apart in the slot):
// v_smem is chunk 2h's address; the first MMA accumulates only if acc.
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, bool acc) {
  const uint32_t vb = desc_lo(v_smem, Cfg<false>::SlotBytes);
  asm volatile(
      "{\n\t.reg .pred p0, p1, e;\n\telect.sync _|e, 0xffffffff;\n\t.reg .b64 b;\n\t.reg .b32 t, y;\n\t"
      "setp.ne.u32 p0, %4, 0;\n\t"
      "setp.eq.u32 p1, %4, %4;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], b, %5, p0;\n\t"
      "add.u32 t, %1, 8;\n\tadd.u32 y, %2, 128;\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], b, %5, p1;\n\t"
      "add.u32 t, %1, 16;\n\tadd.u32 y, %2, 512;\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], b, %5, p1;\n\t"
      "add.u32 t, %1, 24;\n\tadd.u32 y, %2, 640;\n\tmov.b64 b, {y, %3};\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [t], b, %5, p1;\n\t}" ::"r"(d_tmem),
      "r"(p_tmem), "r"(vb), "r"(kDescHi), "r"(acc ? 1u : 0u), "r"(kIdescPV)
      : "memory");
}

// FP8 (whole 128-key tiles, issued by one thread): S = Q (e4m3, 128-byte rows)
// * K^T (e4m3, 64 keys per CTA), 4 pair MMAs of K = 32 (32 bytes of each row
// per step).
__device__ __forceinline__ void issue_qk_f8(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  const uint32_t qa = desc_lo(q_smem, 16), kb = desc_lo(k_smem, 16);
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 a, b;\n\t.reg .b32 x, y;\n\t"
      "setp.ne.u32 p0, %4, %4;\n\t"
      "setp.eq.u32 p1, %4, %4;\n\t"
      "mov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], a, b, %5, p0;\n\t"
      "add.u32 x, %1, 2;\n\tadd.u32 y, %2, 2;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 4;\n\tadd.u32 y, %2, 4;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], a, b, %5, p1;\n\t"
      "add.u32 x, %1, 6;\n\tadd.u32 y, %2, 6;\n\tmov.b64 a, {x, %3};\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], a, b, %5, p1;\n\t}" ::"r"(d_tmem),
      "r"(qa), "r"(kb), "r"(kDescHi), "r"(0u), "r"(kIdescF8)
      : "memory");
}

// FP8: O (+)= P (TMEM, e4m3, four per column) * V (e4m3, K-major: 64 channels
// per CTA, 128-byte rows of keys), 4 pair MMAs of K = 32 keys.
__device__ __forceinline__ void issue_pv_f8(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, bool acc) {
  const uint32_t vb = desc_lo(v_smem, 16);
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 b;\n\t.reg .b32 t, y;\n\t"
      "setp.ne.u32 p0, %4, 0;\n\t"
      "setp.eq.u32 p1, %4, %4;\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [%1], b, %5, p0;\n\t"
      "add.u32 t, %1, 8;\n\tadd.u32 y, %2, 2;\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [t], b, %5, p1;\n\t"
      "add.u32 t, %1, 16;\n\tadd.u32 y, %2, 4;\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [t], b, %5, p1;\n\t"
      "add.u32 t, %1, 24;\n\tadd.u32 y, %2, 6;\n\tmov.b64 b, {y, %3};\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], [t], b, %5, p1;\n\t}" ::"r"(d_tmem),
      "r"(p_tmem), "r"(vb), "r"(kDescHi), "r"(acc ? 1u : 0u), "r"(kIdescF8)
      : "memory");
}

// The MMA warp runs its loop with all 32 lanes (warp-uniform values); each
// tcgen05 instruction is issued by one elected lane.  Commit: arrive on the
// barrier at this offset in both CTAs once the pair MMAs issued so far are done.
__device__ __forceinline__ void commit_pair_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(kPairMask)
      : "memory");
}
__device__ __forceinline__ void commit_pair_local_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// two e4m3 codes of fp32 values (lo in the low byte), round to nearest even, saturating
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// FP8: one query row's 128 scores from TMEM (4 loads of 32 columns); keys past
// the document end (column >= rem) are set to -inf.
__device__ __forceinline__ void load_scores128(uint32_t t_s, uint32_t (&r)[4][32], int rem) {
#pragma unroll
  for (int c = 0; c < 4; ++c) dev::tmem_ld32(t_s + c * 32, r[c]);
  dev::tmem_wait_ld();
  if (rem < kTileRows) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= rem) r[c >> 5][c & 31] = __float_as_uint(-INFINITY);
  }
}

// fp8: 32 accumulator columns times their V channel scales (fp32).
__device__ __forceinline__ void scale_by_channel(uint32_t (&ov)[32], const float* sv) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 s4 = __ldg(reinterpret_cast<const float4*>(sv) + i);
    ov[4 * i] = __float_as_uint(__uint_as_float(ov[4 * i]) * s4.x);
    ov[4 * i + 1] = __float_as_uint(__uint_as_float(ov[4 * i + 1]) * s4.y);
    ov[4 * i + 2] = __float_as_uint(__uint_as_float(ov[4 * i + 2]) * s4.z);
    ov[4 * i + 3] = __float_as_uint(__uint_as_float(ov[4 * i + 3]) * s4.w);
  }
}

// Fused Q prologue for one query row held in shared memory (128-byte swizzled
// K-major tile, two 16 KB halves): RMSNorm with gain and the rot96 rotation,
// in place, with the arithmetic of qk_norm.cuh (the same bits as the
// separate prologue kernel).  Rare (once per row per unit), so kept out of line.
static __device__ __noinline__ void norm_rope_q_row(uint32_t tile, uint32_t r, const float* gain,
                                                    const float2* rope_row, float eps) {
  auto chunk = [&](int c) {  // shared address of dims [8c, 8c + 8) of row r
    return tile + (uint32_t)(c >> 3) * kQHalfBytes + r * 128u + ((((uint32_t)c & 7u) ^ (r & 7u)) << 4);
  };
  auto ld = [&](int c) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(chunk(c)));
    return v;
  };
  auto st = [&](int c, const uint4& v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(chunk(c)), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
  };
  float p[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    float x[8];
    qkn::unpack8(ld(c), x);
    p[c] = qkn::chunk_ss(x);
  }
  const float rr = qkn::inv_rms(qkn::tree16(p), eps);
#pragma unroll 1
  for (int c = 0; c < 6; ++c) {
    float xa[8], xb[8], ya[8], yb[8], cs[8], sn[8];
    qkn::unpack8(ld(c), xa);
    qkn::unpack8(ld(c + 6), xb);
    const float4* ga = reinterpret_cast<const float4*>(gain + 8 * c);
    const float4* gb = reinterpret_cast<const float4*>(gain + 48 + 8 * c);
    const float4 a0 = __ldg(ga), a1 = __ldg(ga + 1), b0 = __ldg(gb), b1 = __ldg(gb + 1);
    const float gav[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float gbv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float4* t = reinterpret_cast<const float4*>(rope_row + 8 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(t + i);  // (cos, sin) of two consecutive angles
      cs[2 * i] = v.x;
      sn[2 * i] = v.y;
      cs[2 * i + 1] = v.z;
      sn[2 * i + 1] = v.w;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ya[e] = qkn::scale_gain(xa[e], rr, gav[e]);
      yb[e] = qkn::scale_gain(xb[e], rr, gbv[e]);
    }
    float oa[8], ob[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      oa[e] = qkn::rot_lo(ya[e], yb[e], cs[e], sn[e]);
      ob[e] = qkn::rot_hi(yb[e], ya[e], cs[e], sn[e]);
    }
    st(c, qkn::pack8(oa));
    st(c + 6, qkn::pack8(ob));
  }
#pragma unroll 1
  for (int c = 12; c < 16; ++c) {
    float x[8];
    qkn::unpack8(ld(c), x);
    const float4* g = reinterpret_cast<const float4*>(gain + 8 * c);
    const float4 g0 = __ldg(g), g1 = __ldg(g + 1);
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = qkn::scale_gain(x[e], rr, gv[e]);
    st(c, qkn::pack8(x));
  }
}

// kFp8: the FP8 variant -- e4m3 Q, K, V (V transposed, keys contiguous) with
// scales (per query row, per key tile, per V channel), kind::f8f6f4 MMAs,
// P rounded to e4m3; everything else as the bf16 kernel.
template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       ForwardArgs a, int o_tma) {
  using C = Cfg<kFp8>;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  const Bars bars{sbase + C::SmemBar};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::SmemMisc + 4);

  const uint32_t warp = dev::warp_id_uniform();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t rank = dev::cluster_ctarank();   // 0: issues the pair's MMAs
  const int pair = (int)(blockIdx.x >> 1);
  // this pair's segments, in order
  const int u_begin = __ldg(a.unit_off + pair), u_end = __ldg(a.unit_off + pair + 1);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) {
      dev::mbar_init(bars.q_full(i), 1);
      // FP8: freed by the MMA issuer after a unit's last QK; bf16: by the
      // O-store thread, once the TMA unit has read the O rows the epilogue
      // staged in the slot
      dev::mbar_init(bars.q_empty(i), 1);
      dev::mbar_init(bars.o_staged(i), 4);
      dev::mbar_init(bars.q_ready(i), 2);           // the Q warp of each CTA of the pair
    }
    for (int s = 0; s < 2; ++s) {
      for (int h = 0; h < 2; ++h) {
        dev::mbar_init(bars.s_ready(s, h), 1);
        dev::mbar_init(bars.p_ready(s, h), 8);      // one arrival per softmax warp of the pair
        dev::mbar_init(bars.pv_done(s, h), 1);
      }
    }
    for (int i = 0; i < kGroups; ++i) {
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
    dev::tmem_alloc_pair(dev::smem_u32(tmem_slot), kTmemCols);
    dev::tmem_relinquish_pair();
  }
  dev::tc_fence_before();
  __syncthreads();
  __syncwarp();
  dev::cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA arrival
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------ TMA producer ----
    if (!kFp8 && lane == 1) {
      // bf16 O stores: as the four softmax warps of a query tile finish a
      // unit's epilogue, send the rows they staged in its Q slot (every warp
      // whose 32 rows lie in the document) with TMA tile stores, wait until
      // they have read the slot, and free it for the Q warp's next load.
      uint32_t use[4] = {0, 0, 0, 0};
      bool ok = true;
      int k = 0;
      for (int u = u_begin; ok && u < u_end; ++u, ++k) {
        const UnitGeom g = unit_geom(a.units, u);
#pragma unroll 1
        for (int s = 0; s < 2 && s < g.n_st; ++s) {
          const int i = 2 * (k & 1) + s;
          ok = dev::mbar_wait(bars.o_staged(i), use[i] & 1, abort_flag, a.err, kTimeoutNs);
          ++use[i];
          if (!ok) break;
          if (o_tma != 0 && g.part < 0) {
            const uint32_t tile = sbase + C::SmemQ + i * C::QTileBytes;
            const int32_t base_row = g.q0 + s * 2 * kTileRows + (int32_t)rank * kTileRows;
            bool any = false;
#pragma unroll 1
            for (int w = 0; w < 4; ++w) {
              const int32_t row0 = base_row + 32 * w;
              if (row0 + 31 >= g.kv1) break;  // (the softmax warps' own test)
              dev::tma_store_2d(&tm_o, tile + 32u * w * 128u, g.head * kHeadDim, row0);
              dev::tma_store_2d(&tm_o, tile + kQHalfBytes + 32u * w * 128u, g.head * kHeadDim + 64, row0);
              any = true;
            }
            if (any) {
              dev::bulk_commit();
              dev::bulk_wait_read_all();
            }
          }
          dev::mbar_arrive(bars.q_empty(i));
        }
      }
      dev::bulk_wait_all();  // the O stores are complete
    }
    if (lane == 0) {
      const uint64_t pol_q = dev::policy_evict_first();
      const uint64_t pol_kv = dev::policy_evict_last();
      uint32_t grp = 0, q_use[4] = {0, 0, 0, 0};
      bool ok = true;
      // FP8: Q tiles of the unit with ordinal k, into buffer k & 1 (the slot
      // is freed by the MMA after the last QK of the unit two before).
      auto load_q = [&](const UnitGeom& g, int k) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          if (!ok || s >= g.n_st) break;
          const int i = 2 * (k & 1) + s;
          ok = dev::mbar_wait(bars.q_empty(i), (q_use[i] & 1) ^ 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          const uint32_t dst = sbase + C::SmemQ + i * C::QTileBytes;
          dev::mbar_arrive_expect_tx(bars.q_full(i), C::QTileBytes);
          const int32_t row = g.q0 + s * 2 * kTileRows + (int32_t)rank * kTileRows;
          dev::tma_load_2d(dst, &tm_q, bars.q_full(i), g.head * 128, row, pol_q);
          if constexpr (!kFp8)
            dev::tma_load_2d(dst + kQHalfBytes, &tm_q, bars.q_full(i), g.head * 128 + 64, row, pol_q);
          ++q_use[i];
        }
      };
      int k = 0;
      for (int u = u_begin; ok && u < u_end; ++u, ++k) {
        const UnitGeom g = unit_geom(a.units, u);
        const bool has_next = u + 1 < u_end;
        // Key/value groups: group 0 is the first unit's first K tile (ring slot
        // 0); group n >= 1 is V(j) with the next K tile -- K(j+1), or the next
        // unit's first K tile -- in slots (2n-1) % kSlots and 2n % kSlots, one
        // full and one empty barrier (index n % kGroups) for both.
        if (k == 0) {
          if constexpr (kFp8) load_q(g, 0);
          if (!ok) break;
          ok = dev::mbar_wait(bars.kv_empty(0), 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          dev::mbar_arrive_expect_tx(bars.kv_full(0), C::SlotBytes);
          load_k_half<kFp8>(sbase + C::SmemKV, &tm_k, bars.kv_full(0), g.head, g.kv0 + g.lo * kTileRows, rank,
                            pol_kv);
          grp = 1;
        }
        for (int j = g.lo; ok && j < g.hi; ++j) {
          bool has_k = j + 1 < g.hi;
          int k_head = g.head;
          int32_t k_row = g.kv0 + (j + 1) * kTileRows;
          if (!has_k && has_next) {
            const UnitGeom n = unit_geom(a.units, u + 1);
            has_k = true;
            k_head = n.head;
            k_row = n.kv0 + n.lo * kTileRows;
          }
          const uint32_t b = grp % kGroups;
          ok = dev::mbar_wait(bars.kv_empty(b), ((grp / kGroups) & 1) ^ 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          dev::mbar_arrive_expect_tx(bars.kv_full(b), has_k ? 2 * C::SlotBytes : C::SlotBytes);
          load_v_half<kFp8>(sbase + C::SmemKV + ((2 * grp - 1) % kSlots) * C::SlotBytes, &tm_v, bars.kv_full(b),
                            g.head, (kFp8 ? g.v_off : g.kv0) + j * kTileRows, rank, pol_kv);
          if (has_k)
            load_k_half<kFp8>(sbase + C::SmemKV + ((2 * grp) % kSlots) * C::SlotBytes, &tm_k, bars.kv_full(b),
                              k_head, k_row, rank, pol_kv);
          ++grp;
          // the next unit's Q tiles, behind this unit's first group
          if constexpr (kFp8)
            if (j == g.lo && has_next) load_q(unit_geom(a.units, u + 1), k + 1);
        }
      }
      if (!ok) {
        // drain: wait (bounded) for every copy this thread issued into the ring and Q
        for (uint32_t r = 1; r <= (uint32_t)kGroups && r <= grp; ++r) {
          const uint32_t n = grp - r;
          dev::mbar_wait_bounded(bars.kv_full(n % kGroups), (n / kGroups) & 1, nullptr, nullptr, kTimeoutNs);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (q_use[i]) dev::mbar_wait_bounded(bars.q_full(i), (q_use[i] - 1) & 1, nullptr, nullptr, kTimeoutNs);
      }
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------- MMA issuer (even CTA, pair) ----
    if constexpr (kFp8) {
      // FP8: whole 128-key tiles (S of a query tile is one barrier phase, P
      // overwrites it), issued by one thread.  Its MMAs are half as long as
      // bf16's, and the halved pipeline measured slower here: the per-half
      // softmax costs would dominate.
      if (lane == 0 && rank == 0) {
        uint32_t vslot = 1, kslot = 2, q_use[4] = {0, 0, 0, 0}, p_it[2] = {0, 0};
        bool ok = true;
        bool issued = false;
        int k = 0;
        for (int u = u_begin; ok && u < u_end; ++u, ++k) {
          const UnitGeom g = unit_geom(a.units, u);
          const uint32_t qb = 2 * (k & 1);
          // Q tiles of this unit, prepared in both CTAs (and, for the first
          // unit, the first K group landed in both)
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (!ok || s >= g.n_st) break;
            ok = dev::mbar_wait(bars.q_ready(qb + s), q_use[qb + s] & 1, abort_flag, a.err, kTimeoutNs);
            ++q_use[qb + s];
          }
          // this unit's first K tile: group 0, or the K half of the previous
          // unit's last group (covered by that unit's last P-ready barrier)
          const uint32_t k0 = k == 0 ? 0u : (kslot >= 2 ? kslot - 2 : kslot + kSlots - 2);
          if (!ok) break;
          dev::tc_fence_after();
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            if (s >= g.n_st) break;
            issue_qk_f8(tmem + s * 128, sbase + C::SmemQ + (qb + s) * C::QTileBytes, sbase + C::SmemKV + k0 * C::SlotBytes);
            dev::mma_commit_pair_mc(bars.s_ready(s, 0), kPairMask);
            if (g.hi - g.lo == 1) dev::mma_commit_pair_mc(bars.q_empty(qb + s), kPairMask);
          }
          issued = true;
          for (int j = g.lo; j < g.hi; ++j) {
            // group grp = V(j) + the next K tile; its arrival in both CTAs is
            // implied by P-ready of query tile 0
            const bool more = j + 1 < g.hi;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              if (s >= g.n_st) break;
              ok = dev::mbar_wait(bars.p_ready(s, 0), p_it[s] & 1, abort_flag, a.err, kTimeoutNs);
              if (!ok) break;
              ++p_it[s];
              dev::tc_fence_after();
              issue_pv_f8(tmem + 256 + s * 128, tmem + s * 128, sbase + C::SmemKV + vslot * C::SlotBytes, j > g.lo);
              if (more) {
                issue_qk_f8(tmem + s * 128, sbase + C::SmemQ + (qb + s) * C::QTileBytes,
                            sbase + C::SmemKV + kslot * C::SlotBytes);
                dev::mma_commit_pair_mc(bars.s_ready(s, 0), kPairMask);
                if (j + 2 == g.hi) dev::mma_commit_pair_mc(bars.q_empty(qb + s), kPairMask);
              } else {
                dev::mma_commit_pair_mc(bars.pv_done(s, 0), kPairMask);  // the unit's O is complete
              }
            }
            if (!ok) break;
            vslot = vslot + 2 >= (uint32_t)kSlots ? vslot + 2 - kSlots : vslot + 2;
            kslot = kslot + 2 >= (uint32_t)kSlots ? kslot + 2 - kSlots : kslot + 2;
          }
        }
        if (!ok && issued) {
          // drain: every MMA issued so far must finish before TMEM is freed
          dev::mma_commit_pair(bars.drain());
          dev::mbar_wait_bounded(bars.drain(), 0, nullptr, nullptr, kTimeoutNs);
        }
      }
    } else if (rank == 0) {
    // bf16: the whole warp runs the loop (its values stay warp-uniform); every
    // tcgen05 MMA and commit is issued by one elected lane.
      // ring slots of the current group's V and K halves: group n uses slots
      // 2n-1 and 2n (mod kSlots), advanced by two per key tile without a division
      uint32_t vslot = 1, kslot = 2, q_use[4] = {0, 0, 0, 0};
      uint32_t p_it[2][2] = {{0, 0}, {0, 0}};
      bool ok = true;
      bool issued = false;
      int k = 0;
      // QK of half h of the key tile in ring slot ks for query tile s (Q slot qs)
      auto qk_half = [&](int s, uint32_t qs, uint32_t ks, int h) {
        const uint32_t d = tmem + s * 128 + h * 64;
        const uint32_t qa = sbase + C::SmemQ + qs * C::QTileBytes;
        const uint32_t kb = sbase + C::SmemKV + ks * C::SlotBytes + h * kHalfKeyRowsBytes;
        issue_qk(d, qa, kb);
        commit_pair_elect(bars.s_ready(s, h));
      };
      // PV of half h of the key tile whose V is in ring slot vs, query tile s
      auto pv_half = [&](int s, uint32_t vs, int h, bool acc) {
        const uint32_t d = tmem + 256 + s * 128, pt = tmem + s * 128 + h * 64;
        const uint32_t vb = sbase + C::SmemKV + vs * C::SlotBytes;
        issue_pv(d, pt, vb + 4096 * h, acc);
      };
      // The first QK (half h) of query tile s of unit gg: Q slot qbase + s (its
      // readiness in both CTAs is awaited before half 0), K in ring slot ks.
      auto first_qk = [&](const UnitGeom& gg, uint32_t qbase, uint32_t ks, int s, int h) {
        if (h == 0) {
          ok = __all_sync(0xffffffffu,
                          dev::mbar_wait(bars.q_ready(qbase + s), q_use[qbase + s] & 1, abort_flag, a.err, kTimeoutNs));
          ++q_use[qbase + s];
          if (!ok) return;
          dev::tc_fence_after();
        }
        qk_half(s, qbase + s, ks, h);
        issued = true;
      };
      for (int u = u_begin; ok && u < u_end; ++u, ++k) {
        const UnitGeom g = unit_geom(a.units, u);
        const uint32_t qb = 2 * (k & 1);
        if (k == 0) {
          // the pair's first unit: its first K tile is group 0 (ring slot 0),
          // and Q-ready also covers that group's arrival in both CTAs
          for (int h = 0; ok && h < 2; ++h)
            for (int s = 0; ok && s < g.n_st; ++s) first_qk(g, qb, 0, s, h);
          if (!ok) break;
        }
        // Per key tile j and half h, for each query tile s: wait for P(s, j, h),
        // then PV(s, j, h) and QK(s, j + 1, h) -- the next key tile's S half
        // goes where P(s, j, h) was, and the softmax works on the other half
        // meanwhile.  In the last key tile all PVs go first (the epilogue
        // waits for them), then the next unit's first QKs.  The next unit's
        // first key tile is the K half of this unit's last group (ring slot
        // kslot in the last key tile); its group is released when the next
        // unit's last query tile sees S of half 1, so that QK comes after
        // every PV of this unit.
        const bool has_next = u + 1 < u_end;
        const UnitGeom gn = unit_geom(a.units, has_next ? u + 1 : u);
        const uint32_t qn = 2 * ((k + 1) & 1);
        const bool two = g.n_st == 2;
        // steady state: key tiles with a next key tile in this unit
        for (int j = g.lo; ok && j + 1 < g.hi; ++j) {
          const bool acc0 = j > g.lo;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              if (s == 1 && !two) break;
              // one lane polls P; the warp follows it
              bool good = true;
              if (lane == 0) good = dev::mbar_wait(bars.p_ready(s, h), p_it[s][h] & 1, abort_flag, a.err, kTimeoutNs);
              ok = __shfl_sync(0xffffffffu, good, 0);
              if (!ok) break;
              ++p_it[s][h];
              dev::tc_fence_after();
              pv_half(s, vslot, h, acc0 || h == 1);
              qk_half(s, qb + s, kslot, h);
            }
            if (!ok) break;
          }
          vslot = vslot + 2 >= (uint32_t)kSlots ? vslot + 2 - kSlots : vslot + 2;
          kslot = kslot + 2 >= (uint32_t)kSlots ? kslot + 2 - kSlots : kslot + 2;
        }
        if (!ok) break;
        // the last key tile: each PV is followed by "PV done" of its half (the
        // epilogue waits for both halves); the next unit's first QKs follow
        // the last PV, so that the epilogue does not wait behind them
        {
          const bool acc0 = g.hi - 1 > g.lo;
          for (int h = 0; ok && h < 2; ++h) {
#pragma unroll 1
            for (int s = 0; s < g.n_st; ++s) {
              ok = __all_sync(0xffffffffu,
                              dev::mbar_wait(bars.p_ready(s, h), p_it[s][h] & 1, abort_flag, a.err, kTimeoutNs));
              if (!ok) break;
              ++p_it[s][h];
              dev::tc_fence_after();
              pv_half(s, vslot, h, acc0 || h == 1);
              commit_pair_elect(bars.pv_done(s, h));
            }
          }
          if (has_next) {
            for (int h = 0; ok && h < 2; ++h)
              for (int s = 0; ok && s < gn.n_st; ++s) first_qk(gn, qn, kslot, s, h);
          }
          vslot = vslot + 2 >= (uint32_t)kSlots ? vslot + 2 - kSlots : vslot + 2;
          kslot = kslot + 2 >= (uint32_t)kSlots ? kslot + 2 - kSlots : kslot + 2;
        }
      }
      if (!ok && issued) {
        // drain: every MMA issued so far must finish before TMEM is freed
        __syncwarp();
        commit_pair_local_elect(bars.drain());
        dev::mbar_wait_bounded(bars.drain(), 0, nullptr, nullptr, kTimeoutNs);
      }
    }
  } else if (warp == kQWarp) {
    // ----------------------------------------------------------- Q warp ----
    // As each of this CTA's Q tiles lands: with the fused Q prologue,
    // normalise and rotate its rows in place (lane l takes rows l, l+32, ...);
    // then report the tile ready to the even CTA.  Before the first unit's
    // first tile, the first K group must have landed too.
    uint32_t q_use[4] = {0, 0, 0, 0};
    bool ok = true;
    const bool fuse_q = a.gain_q != nullptr;
    const uint64_t pol_q = dev::policy_evict_first();
    int k = 0;
    for (int u = u_begin; ok && u < u_end; ++u, ++k) {
      const UnitGeom g = unit_geom(a.units, u);
#pragma unroll 1
      for (int s = 0; s < 2 && s < g.n_st; ++s) {
        const int i = 2 * (k & 1) + s;
        bool good = true;
        if constexpr (!kFp8) {
          // bf16: this warp loads the tile once its slot is free (the
          // O-store thread has sent the previous unit's O rows out of it)
          if (lane == 0) {
            good = dev::mbar_wait(bars.q_empty(i), (q_use[i] & 1) ^ 1, abort_flag, a.err, kTimeoutNs);
            if (good) {
              const uint32_t dst = sbase + C::SmemQ + i * C::QTileBytes;
              const int32_t row = g.q0 + s * 2 * kTileRows + (int32_t)rank * kTileRows;
              dev::mbar_arrive_expect_tx(bars.q_full(i), C::QTileBytes);
              dev::tma_load_2d(dst, &tm_q, bars.q_full(i), g.head * 128, row, pol_q);
              dev::tma_load_2d(dst + kQHalfBytes, &tm_q, bars.q_full(i), g.head * 128 + 64, row, pol_q);
            }
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
        }
        good = dev::mbar_wait(bars.q_full(i), q_use[i] & 1, abort_flag, a.err, kTimeoutNs);
        ++q_use[i];
        if (!kFp8 && good && fuse_q) {
          const int32_t row0 = g.q0 + s * 2 * kTileRows + (int32_t)rank * kTileRows;
          const float* gain = a.gain_q + (int64_t)g.head * a.gain_head_stride;
#pragma unroll 1
          for (uint32_t r = lane; r < (uint32_t)kTileRows; r += 32) {
            const int32_t row = row0 + (int32_t)r;
            if (row < g.kv1)
              norm_rope_q_row(sbase + C::SmemQ + i * C::QTileBytes, r, gain, a.rope + (int64_t)row * kRopeHalf, a.eps);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor cores
        }
        __syncwarp();
        if (good && k == 0 && s == 0 && lane == 0)
          good = dev::mbar_wait(bars.kv_full(0), 0, abort_flag, a.err, kTimeoutNs);
        if (lane == 0) dev::mbar_arrive_cluster(dev::mapa_shared(bars.q_ready(i), 0));
        ok = __all_sync(0xffffffffu, good);
        if (!ok) break;
      }
    }
    if constexpr (!kFp8) {
      if (!ok && lane == 0) {
        // drain: wait (bounded) for the Q copies this warp issued
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (q_use[i]) dev::mbar_wait_bounded(bars.q_full(i), (q_use[i] - 1) & 1, nullptr, nullptr, kTimeoutNs);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax ----
    const int st = warp >> 2;            // query tile of this warpgroup
    const uint32_t row_in_tile = threadIdx.x & 127;
    const uint32_t lane_base = (warp & 3) * 32;
    const uint32_t t_s = tmem + (lane_base << 16) + st * 128;        // S_s / P_s
    const uint32_t t_o = tmem + (lane_base << 16) + 256 + st * 128;  // O_s
    const uint32_t p_ready_remote[2] = {dev::mapa_shared(bars.p_ready(st, 0), 0),
                                        dev::mapa_shared(bars.p_ready(st, 1), 0)};
    const bool lead_lane = (warp & 3) == 0 && lane == 0;             // one lane per warpgroup
    uint32_t s_it[2] = {0, 0};
    uint32_t n_done = 0;                 // units this query tile has finished (PV-done phases per half)
    uint32_t t0 = 0;                     // key tiles the pair has started before this unit
    bool ok = true;
    const float sl2 = a.scale_log2;
    __nv_bfloat16* og = static_cast<__nv_bfloat16*>(a.o);
    // 32-byte output stores when every row start is 32-byte aligned
    const bool o_wide = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0 && (a.o_stride & 15) == 0;
    for (int u = u_begin; ok && u < u_end; ++u) {
      const UnitGeom g = unit_geom(a.units, u);
      const uint32_t t_unit = t0;
      t0 += g.hi - g.lo;
      if (st >= g.n_st) continue;
      const uint32_t q_slot = 2 * ((u - u_begin) & 1) + st;  // this unit's Q tile of this query tile
      // ring bookkeeping by one lane of one warp per CTA
      const bool releases = lead_lane && st == g.n_st - 1;
      const bool checks_kv = lead_lane && st == 0;
      float m_used = -INFINITY, l = 0.f;
      // fp8: this row's q scale (1 for rows past the tensor, never stored)
      float sq_row = 1.f;
      if constexpr (kFp8) {
        const int32_t row = g.q0 + st * 2 * kTileRows + (int32_t)rank * kTileRows + (int32_t)row_in_tile;
        if (row < a.S) sq_row = __ldg(a.sq + (int64_t)g.head * a.S + row);
      }
      if constexpr (kFp8) {
        // FP8: whole 128-key tiles, one S phase per key tile.
        for (int j = g.lo; j < g.hi; ++j) {
          const uint32_t t = t_unit + (j - g.lo);  // the pair's running key-tile count
          // score scale in log2 units: softmax_scale log2(e) times the q-row and key-tile scales
          const float rsc = sl2 * sq_row * __ldg(a.sk + (int64_t)g.head * a.S + g.kv0 + j * kTileRows);
          // (every lane runs the same bounded wait on the same barrier, timer and
          // abort flag in step, so the warp leaves it with one value of ok)
          ok = dev::mbar_wait(bars.s_ready(st, 0), s_it[0] & 1, abort_flag, a.err, kTimeoutNs);
          if (!ok) break;
          ++s_it[0];
          // S of the last query tile is ready: every MMA before it is done, so
          // the group holding K(t) (and V(t-1)) is free in this CTA
          if (releases) dev::mbar_arrive(bars.kv_empty(t % kGroups));
          // test, without blocking, whether the next K/V group has landed; the
          // blocking wait below then only runs if it had not
          const uint32_t kv_bar = bars.kv_full((t + 1) % kGroups), kv_par = ((t + 1) / kGroups) & 1;
          const bool kv_landed = checks_kv && dev::mbar_test_wait(kv_bar, kv_par);
          __syncwarp();  // lanes leave the wait separately; the TMEM loads are warp-collective
          dev::tc_fence_after();
          uint32_t r[4][32];
          float* sv = reinterpret_cast<float*>(&r[0][0]);
          const int rem = g.kv1 - (g.kv0 + j * kTileRows);
          load_scores128(t_s, r, rem);
          // Row max: eight independent chains of 3-input maxima.
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
          for (int c = 16; c < 128; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = dev::max3(mx[i], sv[c + i], sv[c + 8 + i]);
          const float m_new =
              dev::max3(dev::max3(mx[0], mx[1], mx[2]), dev::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * rsc;
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
              dev::fma2(x0, x1, sv[64 * h + 2 * c], sv[64 * h + 2 * c + 1], rsc, rsc, neg, neg);
              const float p0 = dev::ex2_approx(x0), p1 = dev::ex2_approx(x1);
              const int ai = 2 * (c & 3);
              dev::add2(rs8[ai], rs8[ai + 1], rs8[ai], rs8[ai + 1], p0, p1);
              // e4m3, four per column (p <= 2^8 < 448: no scale)
              const uint32_t two = e4m3x2(p0, p1);
              p[c >> 1] = (c & 1) ? (p[c >> 1] | (two << 16)) : two;
            }
            uint32_t p16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) p16[i] = p[i];
            dev::tmem_st16(t_s + 16 * h, p16);
          }
          const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
          l = l * alpha + rs;
          // tcgen05.ld/st are warp-collective (.sync.aligned): the rescale runs
          // for the whole warp when any of its rows needs it (alpha = 1
          // elsewhere); every MMA before the QK just read (PV(t-1) included)
          // has completed.
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
          __syncwarp();
          // the next PV reads V(t) and the QK after it K(t+1): group t+1 must have
          // landed in this CTA before query tile 0 reports P ready
          if (checks_kv && !kv_landed) ok = dev::mbar_wait(kv_bar, kv_par, abort_flag, a.err, kTimeoutNs);
          if (lane == 0) {  // P (and O) of the warp's 32 rows
            if (rank == 0)
              dev::mbar_arrive(bars.p_ready(st, 0));  // the even CTA's own barrier, arrived on locally
            else
              dev::mbar_arrive_cluster(p_ready_remote[0]);
          }
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
      } else {
        // bf16: 64-key halves (see the kernel header).
        for (int j = g.lo; ok && j < g.hi; ++j) {
          const uint32_t t = t_unit + (j - g.lo);  // the pair's running key-tile count
          const float rsc = sl2;  // score scale in log2 units: softmax_scale log2(e)
          const int rem = g.kv1 - (g.kv0 + j * kTileRows);
          const uint32_t kv_bar = bars.kv_full((t + 1) % kGroups), kv_par = ((t + 1) / kGroups) & 1;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // (no lane leaves here: a failed wait only clears ok, and the
            // warp-uniform vote at the end of the half ends the loop)
            ok = dev::mbar_wait(bars.s_ready(st, h), s_it[h] & 1, abort_flag, a.err, kTimeoutNs) && ok;
            ++s_it[h];
            // S half 1 of the last query tile is ready: every MMA before its QK is
            // done, so the group holding K(t) (and V(t-1)) is free in this CTA
            if (releases && h == 1) dev::mbar_arrive(bars.kv_empty(t % kGroups));
            __syncwarp();  // lanes leave the wait separately; the TMEM loads are warp-collective
            dev::tc_fence_after();
            const uint32_t t_sh = t_s + 64 * h;  // this half's S, then its P
            uint32_t r[2][32];
            dev::tmem_ld32(t_sh, r[0]);
            dev::tmem_ld32(t_sh + 32, r[1]);
            dev::tmem_wait_ld();
            float sv[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(r[c >> 5][c & 31]);
            if (rem < kTileRows) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (half_key(c, h) >= rem) sv[c] = -INFINITY;
            }
            // Row max of the half: eight independent chains of 3-input maxima.
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[8 + i]);
#pragma unroll
            for (int c = 16; c < 64; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) mx[i] = dev::max3(mx[i], sv[c + i], sv[c + 8 + i]);
            const float m_new =
                dev::max3(dev::max3(mx[0], mx[1], mx[2]), dev::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * rsc;
            // The reference max only moves when the row max grows by more than
            // 2^8 (then O and l are rescaled; the final O / l is unchanged).
            float alpha = 1.f;
            if (m_new > m_used + kRescaleThreshold) {
              alpha = dev::ex2_approx(m_used - m_new);  // 0 on the first half of a unit (m_used = -inf)
              m_used = m_new;
            }
            const float neg = -m_used;
            float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t p[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              // packed pair arithmetic: one f32x2 FMA for the exponents, one f32x2 add for the sums
              float x0, x1;
              dev::fma2(x0, x1, sv[2 * c], sv[2 * c + 1], rsc, rsc, neg, neg);
              const float p0 = dev::ex2_approx(x0), p1 = dev::ex2_approx(x1);
              const int ai = 2 * (c & 3);
              dev::add2(rs8[ai], rs8[ai + 1], rs8[ai], rs8[ai + 1], p0, p1);
              p[c] = dev::pack_bf16x2(p0, p1);
            }
            dev::tmem_st32(t_sh, p);
            const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
            l = l * alpha + rs;
            // tcgen05.ld/st are warp-collective (.sync.aligned): the rescale runs
            // for the whole warp when any of its rows needs it (alpha = 1
            // elsewhere).  The PV of the previous half (the other half) may
            // still be adding into O (every earlier PV of this tile completed
            // before the QK whose S was just read), so it is awaited first: the
            // QK issued right after it fills the other half's next S, which this
            // thread reads next anyway; in the last key tile no such QK may
            // follow, and "PV done" of half 0 is awaited instead.
            if (!(j == g.lo && h == 0) && __any_sync(0xffffffffu, alpha != 1.f)) {
              if (h == 1 && j + 1 == g.hi)
                ok = dev::mbar_wait(bars.pv_done(st, 0), n_done & 1, abort_flag, a.err, kTimeoutNs) && ok;
              else
                ok = dev::mbar_wait(bars.s_ready(st, 1 - h), s_it[1 - h] & 1, abort_flag, a.err, kTimeoutNs) && ok;
              __syncwarp();
              dev::tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < 8; ++c) {
                uint32_t ov[16];
                dev::tmem_ld16(t_o + c * 16, ov);
                dev::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                dev::tmem_st16(t_o + c * 16, ov);
              }
            }
            dev::tmem_wait_st();
            dev::tc_fence_before();
            __syncwarp();
            // half 0's PV reads V(t) and the QK after it K(t+1): group t+1 must have
            // landed in this CTA before query tile 0 reports that P ready
            // (a blocking wait and the cluster-address arrive measured faster here
            // than FP8's non-blocking test and local arrive)
            if (h == 0 && checks_kv) ok = dev::mbar_wait(kv_bar, kv_par, abort_flag, a.err, kTimeoutNs) && ok;
            if (lane == 0) dev::mbar_arrive_cluster(p_ready_remote[h]);  // P (and O) of the warp's 32 rows
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
          }
        }
      }
      if (!ok) break;
      // the unit's last PVs of this query tile, one per half ("PV done" of a
      // half completes once per unit, after its last key tile's PV; FP8: one,
      // after the unit's last PV)
      ok = dev::mbar_wait(bars.pv_done(st, 0), n_done & 1, abort_flag, a.err, kTimeoutNs) &&
           (kFp8 || dev::mbar_wait(bars.pv_done(st, 1), n_done & 1, abort_flag, a.err, kTimeoutNs));
      ++n_done;
      // every lane of a bf16 warp leaves together (FP8's lanes run the bounded
      // waits in step; its loop is sensitive to code shape)
      if constexpr (kFp8) {
        if (!ok) break;
      } else if (!__all_sync(0xffffffffu, ok)) {
        break;
      }
      __syncwarp();
      dev::tc_fence_after();
      const int32_t local = st * 2 * kTileRows + (int32_t)rank * kTileRows + (int32_t)row_in_tile;
      const int32_t row = g.q0 + local;
      const bool valid = row < g.kv1;
      if (g.part >= 0) {
        // A piece of a unit split along the keys: unnormalised O row, its
        // reference max (log2 units) and sum, for the merge pass.
        // (the partial buffer is a device allocation: its 512-byte rows are 32-byte aligned)
        const size_t slot = (size_t)g.part * kUnitRows + local;
        if constexpr (!kFp8) {
          // bf16: each 32-column chunk of the warp's 32 rows goes through its
          // rows of the unit's Q slot (free: the slot is released only after
          // this warp reports), so that every global store writes whole
          // 128-byte row segments: a store instruction covers 4 rows.
          const uint32_t stage = sbase + C::SmemQ + q_slot * C::QTileBytes + lane_base * 128u;
          const size_t slot0 = (size_t)g.part * kUnitRows + (size_t)(local - (int32_t)lane);
          const int32_t row_first = g.q0 + local - (int32_t)lane;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            dev::tmem_ld32(t_o + c * 32, ov);
            dev::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const uint32_t addr = stage + lane * 128u + ((((uint32_t)e) ^ (lane & 7u)) << 4);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(ov[4 * e]), "r"(ov[4 * e + 1]),
                           "r"(ov[4 * e + 2]), "r"(ov[4 * e + 3])
                           : "memory");
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t r = 4 * i + (lane >> 3), q = lane & 7u;  // row of the warp, 16-byte piece
              uint4 v;
              asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                           : "r"(stage + r * 128u + ((q ^ (r & 7u)) << 4))
                           : "memory");
              if (row_first + (int32_t)r < g.kv1)
                *reinterpret_cast<uint4*>(a.part_o + (slot0 + r) * kHeadDim + c * 32 + 4 * q) = v;
            }
            __syncwarp();
          }
        } else {
          float* dst = a.part_o + slot * kHeadDim;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            dev::tmem_ld32(t_o + c * 32, ov);
            dev::tmem_wait_ld();
            scale_by_channel(ov, a.sv + g.head * kHeadDim + c * 32);
            if (valid) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dev::st_global_v8(dst + c * 32 + e * 8, ov[8 * e], ov[8 * e + 1], ov[8 * e + 2], ov[8 * e + 3],
                                  ov[8 * e + 4], ov[8 * e + 5], ov[8 * e + 6], ov[8 * e + 7]);
            }
          }
        }
        if (valid) a.part_ml[slot] = make_float2(m_used, l);
        if constexpr (!kFp8) {
          __syncwarp();
          if (lane == 0) dev::mbar_arrive(bars.o_staged(q_slot));
        }
        continue;
      }
      const float inv = 1.f / l;
      bool staged = false;
      if constexpr (!kFp8) staged = o_tma != 0 && __all_sync(0xffffffffu, valid);
      if (staged) {
        // The warp's 32 rows, bf16, into its rows of the unit's Q slot (free:
        // every MMA of the unit is done) in the tile's 128-byte swizzled
        // layout; the O-store thread sends them with two TMA stores (dims
        // 0..63, 64..127) of 32 rows each.
        const uint32_t tile = sbase + C::SmemQ + q_slot * C::QTileBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          dev::tmem_ld32(t_o + c * 32, ov);
          dev::tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = dev::pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t cc = 4 * c + e;  // 16-byte chunk of the row
            const uint32_t addr = tile + (cc >> 3) * kQHalfBytes + row_in_tile * 128u + (((cc & 7u) ^ (row_in_tile & 7u)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * e]), "r"(w[4 * e + 1]),
                         "r"(w[4 * e + 2]), "r"(w[4 * e + 3])
                         : "memory");
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(bars.o_staged(q_slot));  // the store thread sends them
      } else {
        __nv_bfloat16* dst = og + (int64_t)row * a.o_stride + g.head * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          dev::tmem_ld32(t_o + c * 32, ov);
          dev::tmem_wait_ld();
          if constexpr (kFp8) scale_by_channel(ov, a.sv + g.head * kHeadDim + c * 32);
          if (valid) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = dev::pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
            if (o_wide) {  // rows and chunks 32-byte aligned: two 32-byte stores per chunk
              dev::st_global_v8(dst + c * 32, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              dev::st_global_v8(dst + c * 32 + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                *reinterpret_cast<uint4*>(dst + c * 32 + e * 8) = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
            }
          }
        }
        if constexpr (!kFp8) {
          __syncwarp();
          if (lane == 0) dev::mbar_arrive(bars.o_staged(q_slot));
        }
      }
      if (valid && a.lse != nullptr)
        a.lse[(int64_t)g.head * a.S + row] = (m_used + __log2f(l)) * 0.6931471805599453f;
    }
  }

  // Neither CTA leaves (or frees the pair's TMEM) while the other may still
  // arrive on its barriers or run MMAs on its shared memory and TMEM.
  dev::tc_fence_before();
  __syncthreads();
  __syncwarp();  // the cluster barrier is warp-collective (.aligned)
  dev::cluster_sync();
  if (warp == kMmaWarp) {
    dev::tc_fence_after();
    dev::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Combines the pieces of units split along the keys: one warp per query row,
// four dims per lane.  With M = max_c m_c (log2 units):
//   o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  lse = (M + log2 l) ln 2.
// At 32 registers a thread, eight blocks fit on an SM, so the rows of a
// typical last round (a few thousand warps) run in one wave.  It is launched
// as a programmatic dependent of the forward: its blocks are scheduled as the
// forward's CTAs leave and wait here for the forward's writes.
__global__ void __launch_bounds__(256, 8) attn_merge_kernel(ForwardArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int mu = warp_global / kUnitRows, r = warp_global % kUnitRows;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the forward is complete and its writes visible
  if (mu >= a.n_merges) return;
  const MergeUnit m = a.merges[mu];
  const int32_t row = m.q_row0 + r;
  if (row >= m.kv_end) return;
  float M = -INFINITY;
#pragma unroll 4
  for (int c = 0; c < m.n_parts; ++c) M = fmaxf(M, a.part_ml[(size_t)(m.part0 + c) * kUnitRows + r].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
#pragma unroll 4
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

// 2D tensor map, 128-byte swizzle: inner extent `inner` elements of `esize`
// bytes (the tile box is 128 bytes wide), `outer` rows `row_bytes` apart.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType type, uint32_t esize, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_rows, std::string* why) {
  auto fn = encode_fn();
  if (fn == nullptr) {
    if (why) *why = "cuTensorMapEncodeTiled is unavailable";
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {128 / esize, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string((int)r);
    return false;
  }
  return true;
}

template <bool kFp8>
cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(attn_fwd_tc_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Cfg<kFp8>::SmemAlloc);
  });
  return attr;
}

template <bool kFp8>
cudaError_t launch_pairs(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                         int o_tma, const ForwardArgs& a, int device, int num_sms, cudaStream_t stream,
                         std::string* why) {
  cudaError_t e = set_smem_attr<kFp8>();
  if (e != cudaSuccess) {
    if (why) *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  (void)device;
  (void)num_sms;
  if (a.n_pairs < 1 || a.unit_off == nullptr) {
    if (why) *why = "the work list has no CTA pairs";
    return cudaErrorInvalidValue;
  }
  attn_fwd_tc_kernel<kFp8><<<2 * a.n_pairs, kThreads, Cfg<kFp8>::SmemAlloc, stream>>>(mq, mk, mv, mo, a, o_tma);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.n_merges == 0) return e;
  const int64_t warps = (int64_t)a.n_merges * kUnitRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_merge_kernel, a);
  if (e != cudaSuccess && why) *why = "the merge launch failed";
  return e;
}

}  // namespace

int forward_slots(int device, int num_sms) {
  // Concurrent CTA pairs: the occupancy of the pair cluster (one CTA per SM),
  // asked once per device; half the SMs if the query fails.  The FP8 kernel
  // has the same threads and registers and less shared memory.
  static int slots[64];
  static std::once_flag once[64];
  if (device < 0 || device >= 64) return num_sms / 2 > 0 ? num_sms / 2 : 1;
  std::call_once(once[device], [device, num_sms] {
    int n = 0;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != device) cudaSetDevice(device);
    if (set_smem_attr<false>() == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (num_sms / 2 > 0 ? num_sms / 2 : 1));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = Cfg<false>::SmemAlloc;
      if (cudaOccupancyMaxActiveClusters(&n, attn_fwd_tc_kernel<false>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    if (prev != device && prev >= 0) cudaSetDevice(prev);
    slots[device] = n > 0 ? n : (num_sms / 2 > 0 ? num_sms / 2 : 1);
  });
  return slots[device];
}

cudaError_t launch_forward(const ForwardArgs& a, int device, int num_sms, cudaStream_t stream, std::string* why) {
  if (a.n_units == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint64_t inner = (uint64_t)a.H * kHeadDim, row = (uint64_t)a.qkv_stride * 2;
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, a.S, row, kTileRows, why) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, a.S, row, kTileRows / 2, why) ||
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, a.S, row, kTileRows, why))
    return cudaErrorInvalidValue;
  // O tiles go out by TMA when its rows allow a tensor map (16-byte aligned
  // base and row stride); otherwise the epilogue stores them directly
  CUtensorMap mo;
  std::memset(&mo, 0, sizeof(mo));
  const bool o_tma = (reinterpret_cast<uintptr_t>(a.o) & 15u) == 0 && (a.o_stride & 7) == 0 &&
                     make_map(&mo, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, a.S, (uint64_t)a.o_stride * 2, 32,
                              nullptr);
  return launch_pairs<false>(mq, mk, mv, mo, o_tma ? 1 : 0, a, device, num_sms, stream, why);
}

cudaError_t launch_forward_fp8(const ForwardArgs& a, int device, int num_sms, cudaStream_t stream,
                               std::string* why) {
  if (a.n_units == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  const uint64_t inner = (uint64_t)a.H * kHeadDim;  // bytes per token row of q8 / k8
  if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner, a.S, inner, kTileRows, why) ||
      !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner, a.S, inner, kTileRows / 2, why) ||
      // transposed V: H * 128 channel rows of S keys, v_row_bytes apart
      !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.v_row_bytes, inner, a.v_row_bytes, kTileRows / 2,
                why))
    return cudaErrorInvalidValue;
  CUtensorMap mo;
  std::memset(&mo, 0, sizeof(mo));
  return launch_pairs<true>(mq, mk, mv, mo, 0, a, device, num_sms, stream, why);
}

}  // namespace h3
