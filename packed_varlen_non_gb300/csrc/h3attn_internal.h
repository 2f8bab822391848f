// Internal declarations shared by the host side of the library (plan builder,
// C-ABI layer) and the kernel launchers.  Nothing here is part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "h3attn.h"

namespace h3 {

constexpr int kHeadDim = 128;
constexpr int kRopeDims = 96;
constexpr int kRopeHalf = 48;       // NeoX pairs (j, j + 48), one angle per pair
constexpr int kAxisFreqs = 16;      // angles per axis: 32 rotated dims per axis / 2
constexpr int kUnitRows = 512;      // query rows per attention work unit (a CTA pair, two 128-row tiles each)

// Device error word values (the word is cleared by h3attn_get_device_error).
constexpr uint32_t kErrNone = 0;
constexpr uint32_t kErrTimeout = 1;

constexpr int kKeyTile = 128;      // key rows per tile

// One attention work segment: up to kUnitRows query rows of one head inside
// one document [kv_begin, kv_end), over that document's key tiles
// [tile_lo, tile_hi) (all of them unless the unit was split along the keys to
// balance the last wave).  part < 0: the segment writes the final output;
// part >= 0: it writes unnormalised partial results to partial slot `part`
// and a merge pass combines the slots of its unit.
struct WorkUnit {
  int32_t q_row0;
  int32_t kv_begin;
  int32_t kv_end;
  int32_t head;
  int32_t tile_lo;
  int32_t tile_hi;
  int32_t part;
  int32_t v_off;   // the document's first key in the FP8 transposed V (16-key aligned)
};
static_assert(sizeof(WorkUnit) == 32, "WorkUnit is read as two 16-byte vectors");

// A unit split along the keys: its partial slots [part0, part0 + n_parts).
struct MergeUnit {
  int32_t q_row0;
  int32_t kv_end;
  int32_t head;
  int32_t part0;
  int32_t n_parts;
  int32_t pad[3];
};
static_assert(sizeof(MergeUnit) == 32, "MergeUnit is read as two 16-byte vectors");

// The attention work units of a packed layout, in list order (longest
// document first, then head, then query rows), and each document's first key
// in the FP8 transposed V (plan.cpp).  Returns an empty string or an error.
std::string build_units(const int32_t* cu, int32_t n_docs, int32_t num_heads, std::vector<WorkUnit>& units,
                        std::vector<int32_t>& v_off, int64_t* v_pad);

// Estimated run time of a segment (plan.cpp), the cost its placement balances.
int64_t segment_cost(const WorkUnit& u);

// Places the n segments on `grid` persistent CTA pairs in list order, each on
// the pair with the least estimated load so far (LPT placement; the list is
// ordered longest document first), and writes them to `out` grouped by pair:
// pair p runs out[unit_off[p] .. unit_off[p + 1]) in order.  Scratch: pair_of
// [n], load and heap [grid]; unit_off has grid + 1 entries.  Returns the number
// of pairs with work (they are pairs 0 .. that number - 1).  No allocation.
int32_t place_pairs(const WorkUnit* segs, size_t n, int grid, WorkUnit* out, int32_t* unit_off,
                    int32_t* pair_of, int64_t* load, int32_t* heap);

// Build the segment list for `grid` persistent CTA pairs: whole units for the
// full rounds, then the last partial round's units split along their key
// tiles into about `grid` pieces, all placed by place_pairs (plan.cpp).
// unit_off gets n_pairs + 1 entries.
void build_segments(const std::vector<WorkUnit>& units, int grid, std::vector<WorkUnit>& segs,
                    std::vector<int32_t>& unit_off, int32_t* n_pairs, std::vector<MergeUnit>& merges,
                    int32_t* n_parts);

struct Plan {
  int device = -1;
  int num_sms = 0;
  int32_t n_docs = 0;
  int32_t num_heads = 0;
  int32_t max_seqlen = 0;
  int64_t S = 0;
  double rope_base = 10000.0;

  std::vector<int32_t> cu_host;      // [n_docs + 1]
  std::vector<double> pos_host;      // [S, 3]
  std::vector<float> rope_host;      // [S, 48, 2] (cos, sin)
  std::vector<WorkUnit> units_host;  // segment list, grouped by CTA pair (see build_segments)
  std::vector<int32_t> unit_off_host;  // [n_pairs + 1]: pair p runs units [unit_off[p], unit_off[p + 1])
  int32_t n_pairs = 0;
  std::vector<MergeUnit> merges_host;
  int32_t n_parts = 0;
  // every document's 128-key tiles: (begin, end, first key in the FP8
  // transposed V, 0); that V gives each document a 16-key aligned start
  std::vector<int4> ktiles_host;
  int64_t v_pad = 0;                 // keys per row of the FP8 transposed V

  int32_t* d_cu = nullptr;
  float2* d_rope = nullptr;          // [S, 48] (cos, sin)
  WorkUnit* d_units = nullptr;       // the segment list, then unit_off (n_pairs + 1 int32)
  int32_t n_units = 0;
  MergeUnit* d_merges = nullptr;
  float* d_part_o = nullptr;         // [n_parts, kUnitRows, 128] unnormalised O
  float2* d_part_ml = nullptr;       // [n_parts, kUnitRows] (running max in log2 units, sum)
  uint32_t* d_err = nullptr;         // device error word
  int4* d_ktiles = nullptr;
};

// Host-side plan construction (plan.cpp); returns an empty string or an error.
// With validate_only, only the document/span checks run (no device needed).
std::string build_plan_host(const h3attn_doc* docs, int32_t n_docs, const h3attn_plan_opts& opts,
                            int grid, Plan& p, bool validate_only = false);

// Error reporting for the C-ABI layer.
h3attn_status fail(h3attn_status s, const char* fmt, ...);
void clear_error();

// Kernel launchers.
struct PrologueArgs {
  const void* q_in;
  const void* k_in;
  void* q_out;
  void* k_out;
  int64_t in_stride;
  int64_t out_stride;
  const float* gain_q;
  const float* gain_k;
  int64_t gain_head_stride;
  const float2* rope;
  int64_t S;
  int32_t H;
  float eps;
};
cudaError_t launch_qk_prologue(const PrologueArgs& a, int num_sms, cudaStream_t stream);

struct ForwardArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t qkv_stride;
  int64_t o_stride;
  int64_t S;
  int32_t H;
  float scale_log2;           // softmax_scale * log2(e)
  const WorkUnit* units;
  int32_t n_units;
  const int32_t* unit_off;    // [n_pairs + 1]: pair p runs units [unit_off[p], unit_off[p + 1])
  int32_t n_pairs;            // CTA pairs launched
  uint32_t* err;
  const MergeUnit* merges;    // may be null when n_merges == 0
  int32_t n_merges;
  float* part_o;
  float2* part_ml;
  // Fused Q prologue (gain_q non-null): q holds the raw queries; the forward
  // applies RMSNorm with gain and the rot96 rotation to each Q tile in shared
  // memory, with the separate prologue's arithmetic.
  const float* gain_q;
  int64_t gain_head_stride;
  float eps;
  const float2* rope;          // [S, 48] (cos, sin)
  // FP8 variant (h3attn_forward_fp8): scales of the e4m3 inputs
  const float* sq;             // [H, S]
  const float* sk;             // [H, S]
  const float* sv;             // [H, 128]
  int64_t v_row_bytes;         // row stride of the transposed V (the plan's v_pad)
};
// Work slots of the forward: CTA pairs that run at the same time on `device`
// (the plan's segment list is balanced for this many).
int forward_slots(int device, int num_sms);
cudaError_t launch_forward(const ForwardArgs& a, int device, int num_sms, cudaStream_t stream,
                           std::string* why);
cudaError_t launch_forward_fp8(const ForwardArgs& a, int device, int num_sms, cudaStream_t stream,
                               std::string* why);

// FP8 (e4m3) quantisation of q-hat, k-hat and v (fp8_quant.cu).
struct Fp8QuantArgs {
  const void* q_hat;
  const void* k_hat;
  const void* v;
  int64_t stride;              // row stride of q-hat, k-hat, v (elements)
  int64_t S;
  int32_t H;
  const int4* tiles;           // (begin, end, V key, 0) of every document's 128-key tiles
  int32_t n_tiles;
  void* q8;                    // [S, H, 128] codes
  void* k8;                    // [S, H, 128] codes
  void* v8t;                   // [H, 128, v_pad] codes, keys contiguous, documents 16-key aligned
  int64_t v_pad;
  float* sq;                   // [H, S]
  float* sk;                   // [H, S] (each token carries its tile's scale)
  float* sv;                   // [H, 128]
};
cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int num_sms, cudaStream_t stream);
// The prologue fused with the q/k quantisation (p: inputs, gains, table; a:
// v and the FP8 outputs), then the v quantisation (fp8_quant.cu).
cudaError_t launch_prologue_fp8(const PrologueArgs& p, const Fp8QuantArgs& a, cudaStream_t stream);

cudaError_t launch_selftest_bounded_wait(uint64_t timeout_ns, uint32_t* d_flag,
                                         cudaStream_t stream);

}  // namespace h3
