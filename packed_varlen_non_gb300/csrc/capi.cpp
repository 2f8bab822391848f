// The C-ABI entry points: argument validation, plan lifetime, launches.
// Every function returns a status and never throws; a failing call leaves a
// message in a thread-local buffer (h3attn_last_error).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "h3attn_internal.h"

namespace h3 {

static thread_local std::string g_last_error;

h3attn_status fail(h3attn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

void clear_error() { g_last_error.clear(); }

}  // namespace h3

using namespace h3;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte extent of a bf16 [S, H, 128] tensor with the given row stride (elements).
struct Extent {
  uintptr_t lo, hi;
};
Extent extent_of(const void* p, int64_t S, int32_t H, int64_t stride) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + (uintptr_t)(((S - 1) * stride + (int64_t)H * kHeadDim) * 2)};
}

// True when two bf16 [S, H, 128] strided tensors can share an element.  With
// equal strides the rows interleave, so compare the column windows modulo the
// stride; with different strides, any byte overlap counts.
bool may_overlap(const void* a, int64_t sa, const void* b, int64_t sb, int64_t S, int32_t H) {
  const Extent ea = extent_of(a, S, H, sa), eb = extent_of(b, S, H, sb);
  if (ea.hi <= eb.lo || eb.hi <= ea.lo) return false;
  if (sa != sb) return true;
  const int64_t width = (int64_t)H * kHeadDim;
  const int64_t delta = ((int64_t)eb.lo - (int64_t)ea.lo) / 2;  // both 16-byte aligned
  int64_t r = delta % sa;
  if (r < 0) r += sa;
  return r < width || r + width > sa;
}

struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  cudaError_t enter(int dev) {
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != dev) {
      e = cudaSetDevice(dev);
      switched = (e == cudaSuccess);
    }
    return e;
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

h3attn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(H3ATTN_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void free_plan_device(Plan* p) {
  if (p->d_cu) cudaFree(p->d_cu);
  if (p->d_rope) cudaFree(p->d_rope);
  if (p->d_units) cudaFree(p->d_units);
  if (p->d_err) cudaFree(p->d_err);
  if (p->d_merges) cudaFree(p->d_merges);
  if (p->d_part_o) cudaFree(p->d_part_o);
  if (p->d_part_ml) cudaFree(p->d_part_ml);
  if (p->d_ktiles) cudaFree(p->d_ktiles);
  p->d_ktiles = nullptr;
  p->d_merges = nullptr;
  p->d_part_o = nullptr;
  p->d_part_ml = nullptr;
  p->d_cu = nullptr;
  p->d_rope = nullptr;
  p->d_units = nullptr;
  p->d_err = nullptr;
}

// Device copy of the plan's unit_off (stored after the segment list).
const int32_t* unit_offsets(const Plan* p) {
  return reinterpret_cast<const int32_t*>(p->d_units + p->units_host.size());
}

h3attn_status check_plan(h3attn_plan_t plan) {
  if (plan == nullptr) return fail(H3ATTN_EINVAL, "plan is NULL");
  return H3ATTN_OK;
}

}  // namespace

struct h3attn_plan : public h3::Plan {};

extern "C" {

const char* h3attn_last_error(void) { return g_last_error.c_str(); }

h3attn_status h3attn_plan_create(const h3attn_doc* docs, int32_t n_docs,
                                 const h3attn_plan_opts* opts, void* cuda_stream,
                                 h3attn_plan_t* out) {
  clear_error();
  if (out == nullptr) return fail(H3ATTN_EINVAL, "out is NULL");
  *out = nullptr;
  if (docs == nullptr) return fail(H3ATTN_EINVAL, "docs is NULL");
  if (opts == nullptr) return fail(H3ATTN_EINVAL, "opts is NULL");
  if (n_docs < 1) return fail(H3ATTN_EINVAL, "n_docs must be >= 1 (got %d)", n_docs);
  if (opts->num_heads < 1) return fail(H3ATTN_EINVAL, "num_heads must be >= 1 (got %d)", opts->num_heads);
  if (opts->head_dim != kHeadDim)
    return fail(H3ATTN_EUNSUPPORTED, "head_dim must be 128 (got %d)", opts->head_dim);
  if (opts->rope_dims != kRopeDims)
    return fail(H3ATTN_EUNSUPPORTED, "rope_dims must be 96 (got %d)", opts->rope_dims);
  if (!std::isfinite(opts->rope_base) || !(opts->rope_base > 1.0))
    return fail(H3ATTN_EINVAL, "rope_base must be finite and > 1");

  // Validate the layout on the host first (no device needed for EINVAL).
  {
    h3attn_plan probe;
    std::string why;
    try {
      why = build_plan_host(docs, n_docs, *opts, 1, probe, /*validate_only=*/true);
    } catch (const std::bad_alloc&) {
      return fail(H3ATTN_ENOMEM, "host allocation failed while building the plan");
    }
    if (!why.empty()) return fail(H3ATTN_EINVAL, "%s", why.c_str());
  }
  h3attn_plan* p = new (std::nothrow) h3attn_plan();
  if (p == nullptr) return fail(H3ATTN_ENOMEM, "host allocation failed");

  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "cudaGetDevice");
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, p->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, p->device);
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (major != 10 || minor != 3) {
    const int dev = p->device;
    delete p;
    return fail(H3ATTN_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, major, minor);
  }
  // the work list is balanced for the forward's persistent CTA pairs
  try {
    build_plan_host(docs, n_docs, *opts, forward_slots(p->device, p->num_sms), *p);
  } catch (const std::bad_alloc&) {
    delete p;
    return fail(H3ATTN_ENOMEM, "host allocation failed while building the plan");
  }

  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const size_t n_cu = p->cu_host.size(), n_rope = (size_t)p->S * kRopeHalf;
  const size_t units_bytes = p->units_host.size() * sizeof(WorkUnit),
               off_bytes = p->unit_off_host.size() * sizeof(int32_t);
  if ((e = cudaMalloc(&p->d_cu, n_cu * sizeof(int32_t))) != cudaSuccess ||
      (e = cudaMalloc(&p->d_rope, n_rope * sizeof(float2))) != cudaSuccess ||
      (e = cudaMalloc(&p->d_units, units_bytes + off_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&p->d_err, 16)) != cudaSuccess ||
      (e = cudaMalloc(&p->d_ktiles, p->ktiles_host.size() * sizeof(int4))) != cudaSuccess ||
      (p->n_parts > 0 &&
       ((e = cudaMalloc(&p->d_merges, p->merges_host.size() * sizeof(MergeUnit))) != cudaSuccess ||
        (e = cudaMalloc(&p->d_part_o, (size_t)p->n_parts * kUnitRows * kHeadDim * sizeof(float))) != cudaSuccess ||
        (e = cudaMalloc(&p->d_part_ml, (size_t)p->n_parts * kUnitRows * sizeof(float2))) != cudaSuccess))) {
    free_plan_device(p);
    delete p;
    return e == cudaErrorMemoryAllocation ? fail(H3ATTN_ENOMEM, "cudaMalloc failed for the plan")
                                          : cuda_fail(e, "cudaMalloc");
  }
  if ((e = cudaMemcpyAsync(p->d_cu, p->cu_host.data(), n_cu * sizeof(int32_t),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(p->d_rope, p->rope_host.data(), n_rope * sizeof(float2),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(p->d_units, p->units_host.data(), units_bytes, cudaMemcpyHostToDevice, st)) !=
          cudaSuccess ||
      (e = cudaMemcpyAsync(p->d_units + p->units_host.size(), p->unit_off_host.data(), off_bytes,
                           cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (p->n_parts > 0 &&
       (e = cudaMemcpyAsync(p->d_merges, p->merges_host.data(), p->merges_host.size() * sizeof(MergeUnit),
                            cudaMemcpyHostToDevice, st)) != cudaSuccess) ||
      (e = cudaMemsetAsync(p->d_err, 0, 16, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(p->d_ktiles, p->ktiles_host.data(), p->ktiles_host.size() * sizeof(int4),
                           cudaMemcpyHostToDevice, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    free_plan_device(p);
    delete p;
    return cuda_fail(e, "plan upload");
  }
  *out = p;
  return H3ATTN_OK;
}

h3attn_status h3attn_plan_destroy(h3attn_plan_t plan) {
  clear_error();
  if (plan == nullptr) return H3ATTN_OK;
  DeviceGuard g;
  g.enter(plan->device);
  cudaDeviceSynchronize();
  free_plan_device(plan);
  delete plan;
  return H3ATTN_OK;
}

h3attn_status h3attn_plan_info(h3attn_plan_t plan, int64_t* total_tokens, int32_t* n_docs,
                               int32_t* max_seqlen, int32_t* num_heads) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (total_tokens) *total_tokens = plan->S;
  if (n_docs) *n_docs = plan->n_docs;
  if (max_seqlen) *max_seqlen = plan->max_seqlen;
  if (num_heads) *num_heads = plan->num_heads;
  return H3ATTN_OK;
}

h3attn_status h3attn_plan_copy_cu_seqlens(h3attn_plan_t plan, int32_t* host_out) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (host_out == nullptr) return fail(H3ATTN_EINVAL, "host_out is NULL");
  // copy back from the device so the check covers the uploaded layout
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e == cudaSuccess)
    e = cudaMemcpy(host_out, plan->d_cu, plan->cu_host.size() * sizeof(int32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e, "copy cu_seqlens");
}

h3attn_status h3attn_plan_copy_positions(h3attn_plan_t plan, double* host_out) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (host_out == nullptr) return fail(H3ATTN_EINVAL, "host_out is NULL");
  std::memcpy(host_out, plan->pos_host.data(), plan->pos_host.size() * sizeof(double));
  return H3ATTN_OK;
}

h3attn_status h3attn_plan_copy_rope_table(h3attn_plan_t plan, float* host_out) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (host_out == nullptr) return fail(H3ATTN_EINVAL, "host_out is NULL");
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e == cudaSuccess)
    e = cudaMemcpy(host_out, plan->d_rope, (size_t)plan->S * kRopeHalf * sizeof(float2),
                   cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e, "copy rope table");
}

h3attn_status h3attn_qk_prologue(h3attn_plan_t plan, const void* q_in, const void* k_in,
                                 int64_t in_row_stride, void* q_out, void* k_out,
                                 int64_t out_row_stride, const float* gain_q,
                                 const float* gain_k, int64_t gain_head_stride, float eps,
                                 void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  // q_in and q_out both NULL: k only (the queries go to h3attn_forward_fused_q)
  const bool with_q = q_in != nullptr || q_out != nullptr;
  if (with_q && (!q_in || !q_out)) return fail(H3ATTN_EINVAL, "q_in and q_out must both be set or both NULL");
  if (!k_in || !k_out || !gain_k || (with_q && !gain_q))
    return fail(H3ATTN_EINVAL, "NULL tensor or gain pointer");
  if (!aligned16(k_in) || !aligned16(k_out) || !aligned16(gain_k) ||
      (with_q && (!aligned16(q_in) || !aligned16(q_out) || !aligned16(gain_q))))
    return fail(H3ATTN_EINVAL, "tensors and gains must be 16-byte aligned");
  const int64_t width = (int64_t)plan->num_heads * kHeadDim;
  if (in_row_stride < width || out_row_stride < width || (in_row_stride % 8) || (out_row_stride % 8))
    return fail(H3ATTN_EINVAL, "row strides must be >= H*128 = %lld and multiples of 8 (got %lld, %lld)",
                (long long)width, (long long)in_row_stride, (long long)out_row_stride);
  if (gain_head_stride != 0 && (gain_head_stride < kHeadDim || (gain_head_stride % 4)))
    return fail(H3ATTN_EINVAL, "gain_head_stride must be 0 or >= 128 and a multiple of 4");
  if (!std::isfinite(eps) || eps < 0.f) return fail(H3ATTN_EINVAL, "eps must be finite and >= 0");
  const int64_t S = plan->S;
  const int32_t H = plan->num_heads;
  // Outputs may alias their own input exactly (in place); no other overlap.
  struct T { const void* p; int64_t s; };
  const T ins[2] = {{q_in, in_row_stride}, {k_in, in_row_stride}};
  const T outs[2] = {{q_out, out_row_stride}, {k_out, out_row_stride}};
  if (with_q && may_overlap(q_out, out_row_stride, k_out, out_row_stride, S, H))
    return fail(H3ATTN_EINVAL, "q_out and k_out overlap");
  for (int o = with_q ? 0 : 1; o < 2; ++o)
    for (int i = with_q ? 0 : 1; i < 2; ++i) {
      const bool same = (outs[o].p == ins[i].p && outs[o].s == ins[i].s && o == i);
      if (!same && may_overlap(outs[o].p, outs[o].s, ins[i].p, ins[i].s, S, H))
        return fail(H3ATTN_EINVAL, "%s_out overlaps %s_in other than exactly in place",
                    o ? "k" : "q", i ? "k" : "q");
    }
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  PrologueArgs a{with_q ? q_in : nullptr, k_in, with_q ? q_out : nullptr, k_out, in_row_stride, out_row_stride,
                 gain_q, gain_k, gain_head_stride, plan->d_rope, S, H, eps};
  e = launch_qk_prologue(a, plan->num_sms, static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e, "qk_prologue launch");
}

static h3attn_status forward_impl(h3attn_plan_t plan, const void* q, const void* k, const void* v,
                                  int64_t qkv_row_stride, void* o, int64_t o_row_stride, float softmax_scale,
                                  float* lse_out, const float* gain_q, int64_t gain_head_stride, float eps,
                                  void* cuda_stream) {
  if (!q || !k || !v || !o) return fail(H3ATTN_EINVAL, "NULL q/k/v/o pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(H3ATTN_EINVAL, "q/k/v/o must be 16-byte aligned");
  if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return fail(H3ATTN_EINVAL, "lse_out must be 4-byte aligned");
  const int64_t width = (int64_t)plan->num_heads * kHeadDim;
  if (qkv_row_stride < width || o_row_stride < width || (qkv_row_stride % 8) || (o_row_stride % 8))
    return fail(H3ATTN_EINVAL, "row strides must be >= H*128 = %lld and multiples of 8 (got %lld, %lld)",
                (long long)width, (long long)qkv_row_stride, (long long)o_row_stride);
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(H3ATTN_EINVAL, "softmax_scale must be finite and > 0");
  const int64_t S = plan->S;
  const int32_t H = plan->num_heads;
  const void* ins[3] = {q, k, v};
  for (int i = 0; i < 3; ++i)
    if (may_overlap(o, o_row_stride, ins[i], qkv_row_stride, S, H))
      return fail(H3ATTN_EINVAL, "o overlaps %c", "qkv"[i]);
  if (lse_out) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(lse_out), hi = lo + (uintptr_t)S * H * 4;
    const Extent eo = extent_of(o, S, H, o_row_stride);
    if (!(hi <= eo.lo || eo.hi <= lo)) return fail(H3ATTN_EINVAL, "lse_out overlaps o");
  }
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  ForwardArgs a{q, k, v, o, lse_out, qkv_row_stride, o_row_stride, S, H,
                softmax_scale * 1.4426950408889634f, plan->d_units, plan->n_units, unit_offsets(plan),
                plan->n_pairs, plan->d_err,
                plan->d_merges, (int32_t)plan->merges_host.size(), plan->d_part_o, plan->d_part_ml,
                gain_q, gain_head_stride, eps, plan->d_rope};
  std::string why;
  e = launch_forward(a, plan->device, plan->num_sms, static_cast<cudaStream_t>(cuda_stream), &why);
  if (e != cudaSuccess) {
    if (!why.empty()) return fail(H3ATTN_ECUDA, "forward: %s", why.c_str());
    return cuda_fail(e, "forward launch");
  }
  return H3ATTN_OK;
}

h3attn_status h3attn_forward(h3attn_plan_t plan, const void* q, const void* k, const void* v,
                             int64_t qkv_row_stride, void* o, int64_t o_row_stride,
                             float softmax_scale, float* lse_out, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  return forward_impl(plan, q, k, v, qkv_row_stride, o, o_row_stride, softmax_scale, lse_out, nullptr, 0, 0.f,
                      cuda_stream);
}

h3attn_status h3attn_forward_fused_q(h3attn_plan_t plan, const void* q_raw, const void* k, const void* v,
                                     int64_t qkv_row_stride, void* o, int64_t o_row_stride,
                                     const float* gain_q, int64_t gain_head_stride, float eps,
                                     float softmax_scale, float* lse_out, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (!gain_q) return fail(H3ATTN_EINVAL, "NULL gain_q");
  if (!aligned16(gain_q)) return fail(H3ATTN_EINVAL, "gain_q must be 16-byte aligned");
  if (gain_head_stride != 0 && (gain_head_stride < kHeadDim || (gain_head_stride % 4)))
    return fail(H3ATTN_EINVAL, "gain_head_stride must be 0 or >= 128 and a multiple of 4");
  if (!std::isfinite(eps) || eps < 0.f) return fail(H3ATTN_EINVAL, "eps must be finite and >= 0");
  return forward_impl(plan, q_raw, k, v, qkv_row_stride, o, o_row_stride, softmax_scale, lse_out, gain_q,
                      gain_head_stride, eps, cuda_stream);
}

// Checks shared by the FP8 quantisation calls: the three bf16 inputs (row
// stride qkv_row_stride) and the six outputs are non-NULL and 16-byte
// aligned, and no output shares bytes with an input or another output.
static h3attn_status check_fp8_io(const Plan* plan, const void* const (&in)[3], int64_t qkv_row_stride, void* q8,
                                  void* k8, void* v8t, float* sq, float* sk, float* sv) {
  if (!in[0] || !in[1] || !in[2] || !q8 || !k8 || !v8t || !sq || !sk || !sv)
    return fail(H3ATTN_EINVAL, "NULL tensor or scale pointer");
  if (!aligned16(in[0]) || !aligned16(in[1]) || !aligned16(in[2]) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(v8t) || !aligned16(sq) || !aligned16(sk) || !aligned16(sv))
    return fail(H3ATTN_EINVAL, "tensors and scales must be 16-byte aligned");
  const int64_t width = (int64_t)plan->num_heads * kHeadDim;
  if (qkv_row_stride < width || (qkv_row_stride % 8))
    return fail(H3ATTN_EINVAL, "row stride must be >= H*128 = %lld and a multiple of 8", (long long)width);
  const int64_t S = plan->S;
  const int32_t H = plan->num_heads;
  const int64_t v_pad = plan->v_pad;
  const uintptr_t in_lo[3] = {reinterpret_cast<uintptr_t>(in[0]), reinterpret_cast<uintptr_t>(in[1]),
                              reinterpret_cast<uintptr_t>(in[2])};
  const uintptr_t in_len = (uintptr_t)(((S - 1) * qkv_row_stride + width) * 2);
  const uintptr_t out_lo[6] = {reinterpret_cast<uintptr_t>(q8), reinterpret_cast<uintptr_t>(k8),
                               reinterpret_cast<uintptr_t>(v8t), reinterpret_cast<uintptr_t>(sq),
                               reinterpret_cast<uintptr_t>(sk), reinterpret_cast<uintptr_t>(sv)};
  const uintptr_t out_len[6] = {(uintptr_t)(S * width), (uintptr_t)(S * width), (uintptr_t)(H * kHeadDim * v_pad),
                                (uintptr_t)(H * S * 4), (uintptr_t)(H * S * 4), (uintptr_t)(H * kHeadDim * 4)};
  for (int o = 0; o < 6; ++o) {
    for (int i = 0; i < 3; ++i)
      if (out_lo[o] < in_lo[i] + in_len && in_lo[i] < out_lo[o] + out_len[o])
        return fail(H3ATTN_EINVAL, "an output overlaps an input");
    for (int o2 = o + 1; o2 < 6; ++o2)
      if (out_lo[o] < out_lo[o2] + out_len[o2] && out_lo[o2] < out_lo[o] + out_len[o])
        return fail(H3ATTN_EINVAL, "two outputs overlap");
  }
  return H3ATTN_OK;
}

h3attn_status h3attn_fp8_quantize(h3attn_plan_t plan, const void* q_hat, const void* k_hat, const void* v,
                                  int64_t qkv_row_stride, void* q8, void* k8, void* v8t, float* sq, float* sk,
                                  float* sv, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  const void* const in[3] = {q_hat, k_hat, v};
  if (h3attn_status s = check_fp8_io(plan, in, qkv_row_stride, q8, k8, v8t, sq, sk, sv)) return s;
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  Fp8QuantArgs a{q_hat, k_hat, v, qkv_row_stride, plan->S, plan->num_heads, plan->d_ktiles,
                 (int32_t)plan->ktiles_host.size(), q8, k8, v8t, plan->v_pad, sq, sk, sv};
  e = launch_fp8_quantize(a, plan->num_sms, static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e, "fp8 quantise launch");
}

h3attn_status h3attn_qk_prologue_fp8(h3attn_plan_t plan, const void* q_in, const void* k_in, const void* v,
                                     int64_t qkv_row_stride, const float* gain_q, const float* gain_k,
                                     int64_t gain_head_stride, float eps, void* q8, void* k8, void* v8t, float* sq,
                                     float* sk, float* sv, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (!gain_q || !gain_k) return fail(H3ATTN_EINVAL, "NULL gain pointer");
  if (!aligned16(gain_q) || !aligned16(gain_k)) return fail(H3ATTN_EINVAL, "gains must be 16-byte aligned");
  if (gain_head_stride != 0 && (gain_head_stride < kHeadDim || (gain_head_stride % 4)))
    return fail(H3ATTN_EINVAL, "gain_head_stride must be 0 or >= 128 and a multiple of 4");
  if (!std::isfinite(eps) || eps < 0.f) return fail(H3ATTN_EINVAL, "eps must be finite and >= 0");
  const void* const in[3] = {q_in, k_in, v};
  if (h3attn_status s = check_fp8_io(plan, in, qkv_row_stride, q8, k8, v8t, sq, sk, sv)) return s;
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  const PrologueArgs p{q_in, k_in, nullptr, nullptr, qkv_row_stride, 0, gain_q, gain_k, gain_head_stride,
                       plan->d_rope, plan->S, plan->num_heads, eps};
  const Fp8QuantArgs a{nullptr, nullptr, v, qkv_row_stride, plan->S, plan->num_heads, plan->d_ktiles,
                       (int32_t)plan->ktiles_host.size(), q8, k8, v8t, plan->v_pad, sq, sk, sv};
  e = launch_prologue_fp8(p, a, static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? H3ATTN_OK : cuda_fail(e, "fp8 prologue launch");
}

h3attn_status h3attn_plan_forward_kernels(h3attn_plan_t plan, int32_t* n_kernels) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (!n_kernels) return fail(H3ATTN_EINVAL, "NULL output pointer");
  *n_kernels = plan->merges_host.empty() ? 1 : 2;
  return H3ATTN_OK;
}

h3attn_status h3attn_work_list_host(const int32_t* cu_seqlens, int32_t n_docs, int32_t num_heads,
                                    int32_t n_pairs, int32_t* units, int64_t units_cap, int32_t* unit_off,
                                    int64_t* n_units, int32_t* n_pairs_used) {
  clear_error();
  if (!cu_seqlens || !n_units || !n_pairs_used) return fail(H3ATTN_EINVAL, "NULL cu_seqlens or output count");
  if (n_docs < 1) return fail(H3ATTN_EINVAL, "n_docs must be >= 1 (got %d)", n_docs);
  if (num_heads < 1) return fail(H3ATTN_EINVAL, "num_heads must be >= 1 (got %d)", num_heads);
  if (n_pairs < 1 || n_pairs > 1024) return fail(H3ATTN_EINVAL, "n_pairs must be in [1, 1024] (got %d)", n_pairs);
  if (cu_seqlens[0] != 0) return fail(H3ATTN_EINVAL, "cu_seqlens[0] must be 0");
  for (int32_t d = 0; d < n_docs; ++d)
    if (cu_seqlens[d + 1] <= cu_seqlens[d])
      return fail(H3ATTN_EINVAL, "document %d is empty or cu_seqlens is not increasing", d);
  try {
    std::vector<WorkUnit> all, segs;
    std::vector<int32_t> v_off, off;
    std::vector<MergeUnit> merges;
    int64_t v_pad = 0;
    int32_t pairs = 0, parts = 0;
    const std::string why = build_units(cu_seqlens, n_docs, num_heads, all, v_off, &v_pad);
    if (!why.empty()) return fail(H3ATTN_EINVAL, "%s", why.c_str());
    build_segments(all, n_pairs, segs, off, &pairs, merges, &parts);
    *n_units = (int64_t)segs.size();
    *n_pairs_used = pairs;
    if (units == nullptr) return H3ATTN_OK;
    if (units_cap < (int64_t)segs.size())
      return fail(H3ATTN_EINVAL, "units_cap %lld < %lld segments", (long long)units_cap, (long long)segs.size());
    std::memcpy(units, segs.data(), segs.size() * sizeof(WorkUnit));
    if (unit_off) std::memcpy(unit_off, off.data(), off.size() * sizeof(int32_t));
  } catch (const std::bad_alloc&) {
    return fail(H3ATTN_ENOMEM, "host allocation failed while building the work list");
  }
  return H3ATTN_OK;
}

h3attn_status h3attn_plan_fp8_v_keys(h3attn_plan_t plan, int64_t* v_keys) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (!v_keys) return fail(H3ATTN_EINVAL, "NULL output pointer");
  *v_keys = plan->v_pad;
  return H3ATTN_OK;
}

h3attn_status h3attn_forward_fp8(h3attn_plan_t plan, const void* q8, const void* k8, const void* v8t,
                                 const float* sq, const float* sk, const float* sv, void* o, int64_t o_row_stride,
                                 float softmax_scale, float* lse_out, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  if (!q8 || !k8 || !v8t || !sq || !sk || !sv || !o) return fail(H3ATTN_EINVAL, "NULL tensor or scale pointer");
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(sq) || !aligned16(sk) || !aligned16(sv) ||
      !aligned16(o))
    return fail(H3ATTN_EINVAL, "tensors and scales must be 16-byte aligned");
  if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return fail(H3ATTN_EINVAL, "lse_out must be 4-byte aligned");
  const int64_t width = (int64_t)plan->num_heads * kHeadDim;
  if (o_row_stride < width || (o_row_stride % 8))
    return fail(H3ATTN_EINVAL, "o_row_stride must be >= H*128 = %lld and a multiple of 8", (long long)width);
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(H3ATTN_EINVAL, "softmax_scale must be finite and > 0");
  const int64_t S = plan->S;
  const int32_t H = plan->num_heads;
  const Extent eo = extent_of(o, S, H, o_row_stride);
  const uintptr_t in_lo[3] = {reinterpret_cast<uintptr_t>(q8), reinterpret_cast<uintptr_t>(k8),
                              reinterpret_cast<uintptr_t>(v8t)};
  const uintptr_t in_len[3] = {(uintptr_t)(S * width), (uintptr_t)(S * width),
                               (uintptr_t)(H * kHeadDim * plan->v_pad)};
  for (int i = 0; i < 3; ++i)
    if (in_lo[i] < eo.hi && eo.lo < in_lo[i] + in_len[i]) return fail(H3ATTN_EINVAL, "o overlaps an input");
  if (lse_out) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(lse_out), hi = lo + (uintptr_t)S * H * 4;
    if (!(hi <= eo.lo || eo.hi <= lo)) return fail(H3ATTN_EINVAL, "lse_out overlaps o");
  }
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  ForwardArgs a{q8, k8, v8t, o, lse_out, width, o_row_stride, S, H,
                softmax_scale * 1.4426950408889634f, plan->d_units, plan->n_units, unit_offsets(plan),
                plan->n_pairs, plan->d_err,
                plan->d_merges, (int32_t)plan->merges_host.size(), plan->d_part_o, plan->d_part_ml,
                nullptr, 0, 0.f, nullptr, sq, sk, sv, plan->v_pad};
  std::string why;
  e = launch_forward_fp8(a, plan->device, plan->num_sms, static_cast<cudaStream_t>(cuda_stream), &why);
  if (e != cudaSuccess) {
    if (!why.empty()) return fail(H3ATTN_ECUDA, "forward: %s", why.c_str());
    return cuda_fail(e, "forward launch");
  }
  return H3ATTN_OK;
}

h3attn_status h3attn_get_device_error(h3attn_plan_t plan, void* cuda_stream) {
  clear_error();
  if (h3attn_status s = check_plan(plan)) return s;
  DeviceGuard g;
  cudaError_t e = g.enter(plan->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "stream synchronize");
  uint32_t word = 0;
  if ((e = cudaMemcpy(&word, plan->d_err, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device error word");
  if (word == kErrNone) return H3ATTN_OK;
  cudaMemset(plan->d_err, 0, sizeof(word));
  if (word == kErrTimeout)
    return fail(H3ATTN_ETIMEOUT, "a bounded device wait ran out; the outputs of that call are invalid");
  return fail(H3ATTN_ECUDA, "device error word 0x%x", word);
}

h3attn_status h3attn_selftest_bounded_wait(uint64_t timeout_ns, void* cuda_stream) {
  clear_error();
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull)
    return fail(H3ATTN_EINVAL, "timeout_ns must be in [1e3, 1e10]");
  uint32_t* d_flag = nullptr;
  cudaError_t e = cudaMalloc(&d_flag, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  uint32_t word = 0;
  if ((e = cudaMemsetAsync(d_flag, 0, sizeof(uint32_t), st)) == cudaSuccess &&
      (e = launch_selftest_bounded_wait(timeout_ns, d_flag, st)) == cudaSuccess &&
      (e = cudaStreamSynchronize(st)) == cudaSuccess)
    e = cudaMemcpy(&word, d_flag, sizeof(word), cudaMemcpyDeviceToHost);
  cudaFree(d_flag);
  if (e != cudaSuccess) return cuda_fail(e, "selftest");
  if (word == kErrTimeout) return fail(H3ATTN_ETIMEOUT, "bounded wait ran out (expected)");
  return fail(H3ATTN_ECUDA, "bounded wait did not report a timeout (word 0x%x)", word);
}

}  // extern "C"
