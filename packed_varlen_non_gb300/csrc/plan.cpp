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
                            int grid, Plan& p, bool validate_only) {
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
  if (validate_only) return "";

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
  // FP8 transposed V: document d's keys start at v_off[d], a multiple of 16
  std::vector<int32_t> v_off(n_docs);
  int64_t v_pad = 0;
  for (int32_t d = 0; d < n_docs; ++d) {
    v_off[d] = (int32_t)v_pad;
    v_pad += (p.cu_host[d + 1] - p.cu_host[d] + 15) / 16 * 16;
  }
  if (v_pad >= (int64_t(1) << 31)) return "too many tokens";
  p.v_pad = v_pad;
  std::vector<WorkUnit> units;
  for (int32_t d : order) {
    const int32_t b = p.cu_host[d], e = p.cu_host[d + 1];
    const int32_t n_kv = (e - b + kKeyTile - 1) / kKeyTile;
    for (int32_t h = 0; h < opts.num_heads; ++h)
      for (int32_t r = b; r < e; r += kUnitRows) units.push_back(WorkUnit{r, b, e, h, 0, n_kv, -1, v_off[d]});
  }
  if (units.size() >= (size_t(1) << 30)) return "too many work units";
  p.ktiles_host.clear();
  for (int32_t d = 0; d < n_docs; ++d)
    for (int32_t t = p.cu_host[d]; t < p.cu_host[d + 1]; t += kKeyTile)
      p.ktiles_host.push_back(int4{t, std::min(t + kKeyTile, p.cu_host[d + 1]), v_off[d] + (t - p.cu_host[d]), 0});
  build_segments(units, grid, p.units_host, p.merges_host, &p.n_parts);
  p.n_units = (int32_t)p.units_host.size();
  return "";
}

// Cost of a unit in tile MMAs: key tiles x active query tiles.
static int64_t unit_cost(const WorkUnit& u) {
  const int64_t tiles = u.tile_hi - u.tile_lo;
  return tiles * ((u.q_row0 + kUnitRows / 2 < u.kv_end) ? 2 : 1);
}

void build_segments(const std::vector<WorkUnit>& units, int grid, std::vector<WorkUnit>& segs,
                    std::vector<MergeUnit>& merges, int32_t* n_parts) {
  // A persistent CTA pair takes segments c, c + grid, c + 2 grid, ...  Whole units
  // fill the first floor(U / grid) rounds in list order (so the CTAs running
  // at one moment share heads and documents, and their keys stay in L2).
  // The L < grid units left for the last round are split along their key
  // tiles into pieces of about equal cost, one piece per pair, so the last
  // round is as long as one piece instead of one whole unit.
  segs.clear();
  merges.clear();
  *n_parts = 0;
  const size_t G = grid > 0 ? (size_t)grid : 1;
  const size_t full = units.size() / G * G;
  segs.assign(units.begin(), units.begin() + full);
  const size_t L = units.size() - full;
  if (L == 0) return;
  std::vector<int32_t> pieces(L, 1);
  int64_t total = 0;
  for (size_t i = 0; i < L; ++i) total += unit_cost(units[full + i]);
  size_t used = L;
  // proportional share of the grid, at most one piece per key tile
  for (size_t i = 0; i < L; ++i) {
    const WorkUnit& u = units[full + i];
    const int64_t want = total > 0 ? (int64_t)(G * unit_cost(u) / total) : 1;
    const int32_t cap = u.tile_hi - u.tile_lo;
    const int32_t n = (int32_t)std::max<int64_t>(1, std::min<int64_t>(want, cap));
    used += n - 1;
    pieces[i] = n;
  }
  // hand out what is left to the units whose pieces are largest
  while (used < G) {
    size_t best = L;
    double best_piece = 0.0;
    for (size_t i = 0; i < L; ++i) {
      const WorkUnit& u = units[full + i];
      if (pieces[i] >= u.tile_hi - u.tile_lo) continue;
      const double piece = (double)unit_cost(u) / pieces[i];
      if (piece > best_piece) {
        best_piece = piece;
        best = i;
      }
    }
    if (best == L) break;
    ++pieces[best];
    ++used;
  }
  for (size_t i = 0; i < L; ++i) {
    const WorkUnit& u = units[full + i];
    const int32_t n = pieces[i], tiles = u.tile_hi - u.tile_lo;
    if (n == 1) {
      segs.push_back(u);
      continue;
    }
    merges.push_back(MergeUnit{u.q_row0, u.kv_end, u.head, *n_parts, n, {0, 0, 0}});
    for (int32_t c = 0; c < n; ++c) {
      WorkUnit piece = u;
      piece.tile_lo = u.tile_lo + (int32_t)((int64_t)tiles * c / n);
      piece.tile_hi = u.tile_lo + (int32_t)((int64_t)tiles * (c + 1) / n);
      piece.part = (*n_parts)++;
      segs.push_back(piece);
    }
  }
}

}  // namespace h3
