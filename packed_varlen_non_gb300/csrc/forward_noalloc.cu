// h3attn_forward_noalloc: the packed varlen forward without a plan and
// without any device allocation.
//
// Who needs this: callers that are not allowed to allocate device memory
// themselves or through this library -- for example a host application whose
// device memory is owned by a framework's pool or arena (an inference engine
// plugin, a serving runtime that pre-reserves all memory at start-up), or a
// latency-critical loop where a cudaMalloc would synchronise the device.
// h3attn_plan_create allocates the plan's device arrays, so such callers
// cannot use h3attn_forward; this entry point builds the same work list on
// the host and keeps it, with the kernel's error word, in one file-scope
// device array instead.
//
// The array is a static __device__ object: every GPU that loads the library
// holds it (16 B + 4 KiB of per-pair offsets + 32768 x 32 B = 1 MiB + 4 KiB +
// 16 B) until the process exits, all calls share it, and it keeps the last
// call's contents.  In host code its name is only a
// host-side stand-in, so the device address is taken once per device with
// cudaGetSymbolAddress (on the first call on that device, with the device
// current) and passed to the kernel.
#include <algorithm>
#include <mutex>
#include <string>

#include "h3attn_internal.h"

namespace h3 {

namespace {

constexpr int32_t kNoAllocMaxUnits = 32768;  // work units of up to kUnitRows query rows x one head
constexpr int32_t kNoAllocMaxPairs = 1024;   // CTA pairs the offsets can describe
constexpr int32_t kOffsetVecs = (kNoAllocMaxPairs + 1 + 3) / 4;  // int4 holding the offsets
constexpr int kMaxDevices = 64;

// [0]: device error word (cleared before every launch); [1, 1 + kOffsetVecs):
// per-pair offsets into the work list (int32, pairs + 1 of them); then the
// work list (one 32-byte record, two int4, per unit), grouped by pair.
static __device__ __align__(256) int4 g_noalloc_scratch[1 + kOffsetVecs + 2 * kNoAllocMaxUnits];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once).
cudaError_t scratch_on_device(int dev, int4** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<int4*>(g_scratch_ptr[dev]);
  return cudaSuccess;
}

// Host staging of the work list (pageable; cudaMemcpyAsync from pageable
// memory returns once the bytes are staged, so the buffer can be refilled by
// the next call).  Guarded by a mutex held until the kernel is enqueued, so
// host threads do not interleave their copies and launches.
std::mutex g_stage_mutex;
WorkUnit g_stage[kNoAllocMaxUnits];
int32_t g_order[kNoAllocMaxUnits];
// the image of the device array after its error word: offsets, then the placed work list
struct StageImage {
  int32_t unit_off[kOffsetVecs * 4];
  WorkUnit units[kNoAllocMaxUnits];
};
static_assert(sizeof(StageImage) == sizeof(int4) * (kOffsetVecs + 2 * kNoAllocMaxUnits), "layout");
StageImage g_image;
int32_t g_pair_of[kNoAllocMaxUnits];
int64_t g_load[kNoAllocMaxPairs];
int32_t g_heap[kNoAllocMaxPairs];

}  // namespace

}  // namespace h3

using namespace h3;

extern "C" h3attn_status h3attn_forward_noalloc(const int32_t* cu_seqlens, int32_t n_docs,
                                                int32_t num_heads, const void* q, const void* k,
                                                const void* v, int64_t qkv_row_stride, void* o,
                                                int64_t o_row_stride, float softmax_scale,
                                                float* lse_out, void* cuda_stream) {
  clear_error();
  if (cu_seqlens == nullptr) return fail(H3ATTN_EINVAL, "cu_seqlens is NULL");
  if (n_docs < 1) return fail(H3ATTN_EINVAL, "n_docs must be >= 1 (got %d)", n_docs);
  if (num_heads < 1) return fail(H3ATTN_EINVAL, "num_heads must be >= 1 (got %d)", num_heads);
  if (!q || !k || !v || !o) return fail(H3ATTN_EINVAL, "NULL q/k/v/o pointer");
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o))
    return fail(H3ATTN_EINVAL, "q/k/v/o must be 16-byte aligned");
  if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return fail(H3ATTN_EINVAL, "lse_out must be 4-byte aligned");
  const int64_t width = (int64_t)num_heads * kHeadDim;
  if (qkv_row_stride < width || o_row_stride < width || (qkv_row_stride % 8) || (o_row_stride % 8))
    return fail(H3ATTN_EINVAL, "row strides must be >= H*128 = %lld and multiples of 8",
                (long long)width);
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale || softmax_scale > 3.0e38f)
    return fail(H3ATTN_EINVAL, "softmax_scale must be finite and > 0");
  if (cu_seqlens[0] != 0) return fail(H3ATTN_EINVAL, "cu_seqlens[0] must be 0");
  int64_t n_units = 0;
  for (int32_t d = 0; d < n_docs; ++d) {
    const int64_t len = (int64_t)cu_seqlens[d + 1] - cu_seqlens[d];
    if (len < 1) return fail(H3ATTN_EINVAL, "document %d is empty or cu_seqlens is not increasing", d);
    n_units += (len + kUnitRows - 1) / kUnitRows * num_heads;
  }
  if (n_units > kNoAllocMaxUnits)
    return fail(H3ATTN_EINVAL,
                "this layout needs %lld work units; the allocation-free forward holds at most %d "
                "(use h3attn_plan_create + h3attn_forward)",
                (long long)n_units, kNoAllocMaxUnits);
  const int64_t S = cu_seqlens[n_docs];
  {
    // o must not share a byte range with q, k or v (conservative, no column analysis)
    auto lo = [](const void* p) { return reinterpret_cast<uintptr_t>(p); };
    auto hi = [&](const void* p, int64_t st) {
      return lo(p) + (uintptr_t)(((S - 1) * st + width) * 2);
    };
    const void* ins[3] = {q, k, v};
    for (int i = 0; i < 3; ++i)
      if (!(hi(o, o_row_stride) <= lo(ins[i]) || hi(ins[i], qkv_row_stride) <= lo(o)))
        return fail(H3ATTN_EINVAL, "o shares bytes with %c", "qkv"[i]);
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(H3ATTN_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(H3ATTN_EUNSUPPORTED, "device index %d", dev);
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(H3ATTN_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                major, minor);
  int4* scratch = nullptr;
  if ((e = scratch_on_device(dev, &scratch)) != cudaSuccess)
    return fail(H3ATTN_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));

  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // The lock is held from staging the work list until the kernel is enqueued:
  // two host threads sharing a stream then enqueue (copy, kernel) pairs that
  // never interleave, so each kernel reads its own list.
  std::lock_guard<std::mutex> lock(g_stage_mutex);
  int32_t n_pairs = 0;
  {
    // Same work-list order as a plan: longest documents first, then head, then query tile.
    // (each document contributes at least one unit, so n_docs <= n_units <= the buffer size)
    for (int32_t d = 0; d < n_docs; ++d) g_order[d] = d;
    std::sort(g_order, g_order + n_docs, [cu_seqlens](int32_t x, int32_t y) {
      const int32_t lx = cu_seqlens[x + 1] - cu_seqlens[x], ly = cu_seqlens[y + 1] - cu_seqlens[y];
      return lx != ly ? lx > ly : x < y;
    });
    // whole units only (no key-range split, so no partial buffers are needed),
    // placed on the pairs as a plan places them
    int32_t nu = 0;
    for (int32_t i = 0; i < n_docs; ++i) {
      const int32_t b = cu_seqlens[g_order[i]], en = cu_seqlens[g_order[i] + 1];
      const int32_t n_kv = (en - b + kKeyTile - 1) / kKeyTile;
      for (int32_t h = 0; h < num_heads; ++h)
        for (int32_t r = b; r < en; r += kUnitRows) g_stage[nu++] = WorkUnit{r, b, en, h, 0, n_kv, -1, 0};
    }
    const int slots = forward_slots(dev, sms);
    const int grid = slots < kNoAllocMaxPairs ? slots : kNoAllocMaxPairs;
    n_pairs = place_pairs(g_stage, (size_t)nu, grid, g_image.units, g_image.unit_off, g_pair_of, g_load, g_heap);
    const size_t bytes = sizeof(int4) * kOffsetVecs + sizeof(WorkUnit) * (size_t)nu;
    if ((e = cudaMemsetAsync(scratch, 0, sizeof(int4), st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(scratch + 1, &g_image, bytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
      return fail(H3ATTN_ECUDA, "staging the work list: %s", cudaGetErrorString(e));
  }
  ForwardArgs a{q, k, v, o, lse_out, qkv_row_stride, o_row_stride, S, num_heads,
                softmax_scale * 1.4426950408889634f,
                reinterpret_cast<const WorkUnit*>(scratch + 1 + kOffsetVecs), (int32_t)n_units,
                reinterpret_cast<const int32_t*>(scratch + 1), n_pairs, reinterpret_cast<uint32_t*>(scratch),
                nullptr, 0, nullptr, nullptr};
  std::string why;
  e = launch_forward(a, dev, sms, st, &why);
  if (e != cudaSuccess)
    return fail(H3ATTN_ECUDA, "forward: %s", why.empty() ? cudaGetErrorString(e) : why.c_str());
  return H3ATTN_OK;
}
