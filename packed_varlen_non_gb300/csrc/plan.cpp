// Host-side plan builder: cu_seqlens, the fp64 (t, h, w) position grid, the
// fp32 cos/sin table and the attention work list.
//
// Pages: vllm.cpp PR #26 "feat(minimax-h3)", PR description -- documents are
// packed back to back and delimited by cu_seqlens; the fp64 grid that feeds
// the rotary embedding is gated bit-exact, which requires upstream's
// arithmetic order (a linspace without endpoint computes i*step + start);
// "The device-resident forward (W2b)" -- the rotary angles come off the fp64
// grid and feed a per-row cos/sin cache built on the host.  "h3-spark" model
// card, "What this config does" -- rope caches are step-invariant, so the plan
// is built once per request.
//
// This file must be compiled with -ffp-contract=off: a fused multiply-add in
// i*step + start would change the last bit of the grid.
#include <cmath>
#include <cstring>
#include <algorithm>

#include "h3attn_internal.h"

namespace h3 {

static bool finite3(const double* a) {
  return std::isfinite(a[0]) && std::isfinite(a[1]) && std::isfinite(a[2]);
}

std::string build_plan_host(const h3attn_doc* docs, int32_t n_docs, const h3attn_plan_opts& opts,
                            Plan& p) {
  p.n_docs = n_docs;
  p.num_heads = opts.num_heads;
  p.rope_base = opts.rope_base;
  p.cu_host.assign(1, 0);
  int64_t S = 0;
  int32_t max_len = 0;
  for (int32_t d = 0; d < n_docs; ++d) {
    const h3attn_doc& doc = docs[d];
    if (doc.n_spans < 1 || doc.spans == nullptr) return "document " + std::to_string(d) + " has no spans";
    int64_t len = 0;
    for (int32_t s = 0; s < doc.n_spans; ++s) {
      const h3attn_span& sp = doc.spans[s];
      if (sp.n_t < 1 || sp.n_h < 1 || sp.n_w < 1)
        return "document " + std::to_string(d) + " span " + std::to_string(s) + " has a non-positive extent";
      if (!finite3(sp.start) || !finite3(sp.step))
        return "document " + std::to_string(d) + " span " + std::to_string(s) + " has a non-finite start or step";
      len += (int64_t)sp.n_t * sp.n_h * sp.n_w;
      if (len >= (int64_t(1) << 31)) return "document too long";
    }
    S += len;
    if (S >= (int64_t(1) << 31)) return "total tokens S must be < 2^31";
    max_len = std::max<int32_t>(max_len, (int32_t)len);
    p.cu_host.push_back((int32_t)S);
  }
  p.S = S;
  p.max_seqlen = max_len;

  // fp64 grid: per span, t-major then h, w fastest; one rounded product, one rounded sum.
  p.pos_host.resize((size_t)S * 3);
  size_t row = 0;
  for (int32_t d = 0; d < n_docs; ++d) {
    for (int32_t s = 0; s < docs[d].n_spans; ++s) {
      const h3attn_span& sp = docs[d].spans[s];
      for (int32_t it = 0; it < sp.n_t; ++it)
        for (int32_t ih = 0; ih < sp.n_h; ++ih)
          for (int32_t iw = 0; iw < sp.n_w; ++iw) {
            const double idx[3] = {(double)it, (double)ih, (double)iw};
            for (int a = 0; a < 3; ++a) {
              const double prod = idx[a] * sp.step[a];
              p.pos_host[row * 3 + a] = prod + sp.start[a];
            }
            ++row;
          }
    }
  }

  // cos/sin table: angle a*16 + k = pos[a] * base^(-2k/32), in fp64, stored as fp32 pairs.
  double inv_freq[kAxisFreqs];
  const double d_axis = (double)(kRopeDims / 3);
  for (int k = 0; k < kAxisFreqs; ++k) inv_freq[k] = std::pow(opts.rope_base, -(2.0 * k) / d_axis);
  p.rope_host.resize((size_t)S * kRopeHalf * 2);
  for (int64_t i = 0; i < S; ++i) {
    for (int a = 0; a < 3; ++a) {
      for (int k = 0; k < kAxisFreqs; ++k) {
        const double th = p.pos_host[i * 3 + a] * inv_freq[k];
        const size_t o = ((size_t)i * kRopeHalf + a * kAxisFreqs + k) * 2;
        p.rope_host[o] = (float)std::cos(th);
        p.rope_host[o + 1] = (float)std::sin(th);
      }
    }
  }

  // Work list: documents longest first (their units cost most), then head,
  // then query tile.  Consecutive units share (document, head), so the CTAs
  // running at the same moment read the same keys and values through L2.
  std::vector<int32_t> order(n_docs);
  for (int32_t d = 0; d < n_docs; ++d) order[d] = d;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return (p.cu_host[a + 1] - p.cu_host[a]) > (p.cu_host[b + 1] - p.cu_host[b]);
  });
  p.units_host.clear();
  for (int32_t d : order) {
    const int32_t b = p.cu_host[d], e = p.cu_host[d + 1];
    for (int32_t h = 0; h < opts.num_heads; ++h)
      for (int32_t r = b; r < e; r += kUnitRows) p.units_host.push_back(WorkUnit{r, b, e, h});
  }
  if (p.units_host.size() >= (size_t(1) << 31)) return "too many work units";
  p.n_units = (int32_t)p.units_host.size();
  return "";
}

}  // namespace h3
