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

std::string build_units(const int32_t* cu, int32_t n_docs, int32_t num_heads, std::vector<WorkUnit>& units,
                        std::vector<int32_t>& v_off, int64_t* v_pad) {
  // Work list: documents longest first (their units cost most), then head,
  // then query tile.  Consecutive units share (document, head), so the CTAs
  // running at the same moment read the same keys and values through L2.
  std::vector<int32_t> order(n_docs);
  for (int32_t d = 0; d < n_docs; ++d) order[d] = d;
  std::stable_sort(order.begin(), order.end(),
                   [cu](int32_t a, int32_t b) { return (cu[a + 1] - cu[a]) > (cu[b + 1] - cu[b]); });
  // FP8 transposed V: document d's keys start at v_off[d], a multiple of 16
  v_off.assign(n_docs, 0);
  int64_t pad = 0;
  for (int32_t d = 0; d < n_docs; ++d) {
    v_off[d] = (int32_t)pad;
    pad += (cu[d + 1] - cu[d] + 15) / 16 * 16;
  }
  if (pad >= (int64_t(1) << 31)) return "too many tokens";
  *v_pad = pad;
  units.clear();
  for (int32_t d : order) {
    const int32_t b = cu[d], e = cu[d + 1];
    const int32_t n_kv = (e - b + kKeyTile - 1) / kKeyTile;
    for (int32_t h = 0; h < num_heads; ++h)
      for (int32_t r = b; r < e; r += kUnitRows) {
        units.push_back(WorkUnit{r, b, e, h, 0, n_kv, -1, v_off[d]});
        if (units.size() >= (size_t(1) << 30)) return "too many work units";
      }
  }
  return "";
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

  std::vector<WorkUnit> units;
  std::vector<int32_t> v_off;
  const std::string why = build_units(p.cu_host.data(), n_docs, opts.num_heads, units, v_off, &p.v_pad);
  if (!why.empty()) return why;
  p.ktiles_host.clear();
  for (int32_t d = 0; d < n_docs; ++d)
    for (int32_t t = p.cu_host[d]; t < p.cu_host[d + 1]; t += kKeyTile)
      p.ktiles_host.push_back(int4{t, std::min(t + kKeyTile, p.cu_host[d + 1]), v_off[d] + (t - p.cu_host[d]), 0});
  build_segments(units, grid, p.units_host, p.unit_off_host, &p.n_pairs, p.merges_host, &p.n_parts);
  p.n_units = (int32_t)p.units_host.size();
  return "";
}

// Estimated run time of a segment, in key-tile periods: one per key tile and
// one for its start and epilogue.  A segment with only one active query tile
// (at most 256 rows of the document left) costs about as much per key tile as
// one with two: the period is set by the chain softmax -> PV -> QK of each
// tile, which the second tile only overlaps.
int64_t segment_cost(const WorkUnit& u) { return (int64_t)(u.tile_hi - u.tile_lo) + 1; }

int32_t place_pairs(const WorkUnit* segs, size_t n, int grid, WorkUnit* out, int32_t* unit_off,
                    int32_t* pair_of, int64_t* load, int32_t* heap) {
  const int G = grid > 0 ? grid : 1;
  // min-heap of pair indices ordered by (load, index); all loads start at 0,
  // so the identity order is already a heap
  for (int p = 0; p < G; ++p) {
    load[p] = 0;
    heap[p] = p;
  }
  auto before = [load](int32_t a, int32_t b) { return load[a] != load[b] ? load[a] < load[b] : a < b; };
  for (size_t i = 0; i < n; ++i) {
    const int32_t p = heap[0];
    pair_of[i] = p;
    load[p] += segment_cost(segs[i]);
    for (int c = 0;;) {
      const int l = 2 * c + 1, r = l + 1;
      int m = c;
      if (l < G && before(heap[l], heap[m])) m = l;
      if (r < G && before(heap[r], heap[m])) m = r;
      if (m == c) break;
      std::swap(heap[c], heap[m]);
      c = m;
    }
  }
  // pair-major order (a counting sort that keeps each pair's list order);
  // heap[] becomes the fill cursor of each pair
  for (int p = 0; p <= G; ++p) unit_off[p] = 0;
  for (size_t i = 0; i < n; ++i) ++unit_off[pair_of[i] + 1];
  for (int p = 0; p < G; ++p) unit_off[p + 1] += unit_off[p];
  for (int p = 0; p < G; ++p) heap[p] = unit_off[p];
  for (size_t i = 0; i < n; ++i) out[heap[pair_of[i]]++] = segs[i];
  // every placement adds a positive cost and ties go to the lower index, so
  // the first min(n, G) segments open pairs 0, 1, ... in turn: the pairs with
  // work are exactly the leading ones
  int32_t used = 0;
  while (used < G && unit_off[used + 1] > unit_off[used]) ++used;
  return used;
}

void build_segments(const std::vector<WorkUnit>& units, int grid, std::vector<WorkUnit>& segs,
                    std::vector<int32_t>& unit_off, int32_t* n_pairs, std::vector<MergeUnit>& merges,
                    int32_t* n_parts) {
  // The units of the first floor(U / grid) rounds are placed whole.  The
  // L < grid units left over are split along their key tiles into pieces of
  // about equal cost (about grid pieces in all), which are placed after them,
  // so the last round ends at about the same time on every pair.  Placement
  // is LPT in list order (place_pairs).
  merges.clear();
  *n_parts = 0;
  const size_t G = grid > 0 ? (size_t)grid : 1;
  const size_t full = units.size() / G * G;
  std::vector<WorkUnit> cand(units.begin(), units.begin() + full);
  const size_t L = units.size() - full;
  auto work = [](const WorkUnit& u) { return segment_cost(u) - 1; };
  if (L > 0) {
    std::vector<int32_t> pieces(L, 1);
    int64_t total = 0;
    for (size_t i = 0; i < L; ++i) total += work(units[full + i]);
    size_t used = L;
    // proportional share of the grid, at most one piece per key tile
    for (size_t i = 0; i < L; ++i) {
      const WorkUnit& u = units[full + i];
      const int64_t want = total > 0 ? (int64_t)(G * work(u) / total) : 1;
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
        const double piece = (double)work(u) / pieces[i];
        if (piece > best_piece) {
          best_piece = piece;
          best = i;
        }
      }
      if (best == L) break;
      ++pieces[best];
      ++used;
    }
    std::vector<WorkUnit> tail;
    for (size_t i = 0; i < L; ++i) {
      const WorkUnit& u = units[full + i];
      const int32_t n = pieces[i], tiles = u.tile_hi - u.tile_lo;
      if (n == 1) {
        tail.push_back(u);
        continue;
      }
      merges.push_back(MergeUnit{u.q_row0, u.kv_end, u.head, *n_parts, n, {0, 0, 0}});
      for (int32_t c = 0; c < n; ++c) {
        WorkUnit piece = u;
        piece.tile_lo = u.tile_lo + (int32_t)((int64_t)tiles * c / n);
        piece.tile_hi = u.tile_lo + (int32_t)((int64_t)tiles * (c + 1) / n);
        piece.part = (*n_parts)++;
        tail.push_back(piece);
      }
    }
    cand.insert(cand.end(), tail.begin(), tail.end());
  }
  segs.resize(cand.size());
  unit_off.assign(G + 1, 0);
  std::vector<int32_t> pair_of(cand.size()), heap(G);
  std::vector<int64_t> load(G);
  *n_pairs = place_pairs(cand.data(), cand.size(), (int)G, segs.data(), unit_off.data(), pair_of.data(),
                         load.data(), heap.data());
  unit_off.resize((size_t)*n_pairs + 1);
}

}  // namespace h3
