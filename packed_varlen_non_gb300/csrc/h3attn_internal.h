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
constexpr int kUnitRows = 256;      // query rows per attention work unit (two 128-row tiles)

// Device error word values (the word is cleared by h3attn_get_device_error).
constexpr uint32_t kErrNone = 0;
constexpr uint32_t kErrTimeout = 1;

// One attention work unit: up to kUnitRows query rows of one head inside one
// document; the key/value range is the whole document [kv_begin, kv_end).
struct WorkUnit {
  int32_t q_row0;
  int32_t kv_begin;
  int32_t kv_end;
  int32_t head;
};
static_assert(sizeof(WorkUnit) == 16, "WorkUnit is read as one 16-byte vector");

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
  std::vector<WorkUnit> units_host;  // work list, longest documents first

  int32_t* d_cu = nullptr;
  float2* d_rope = nullptr;          // [S, 48] (cos, sin)
  WorkUnit* d_units = nullptr;
  int32_t n_units = 0;
  uint32_t* d_err = nullptr;         // device error word
};

// Host-side plan construction (plan.cpp); returns an empty string or an error.
std::string build_plan_host(const h3attn_doc* docs, int32_t n_docs, const h3attn_plan_opts& opts,
                            Plan& p);

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
  uint32_t* err;
};
cudaError_t launch_forward(const ForwardArgs& a, int num_sms, cudaStream_t stream,
                           std::string* why);

cudaError_t launch_selftest_bounded_wait(uint64_t timeout_ns, uint32_t* d_flag,
                                         cudaStream_t stream);

}  // namespace h3
