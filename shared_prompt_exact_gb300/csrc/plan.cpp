// plan.cpp -- host planner for the packed DualKV layout: index builder and the
// work lists of the forward, dQ and dK/dV kernels.
#include "plan.h"

#include <algorithm>
#include <climits>

namespace dkv {

const char* validate_layout(int P, int N, const int32_t* off, int Hq, int Hkv, int D) {
  if (P < 0) return "P must be >= 0";
  if (N < 1) return "N must be >= 1";
  if (!off) return "R_offsets is null";
  if (off[0] != 0) return "R_offsets[0] must be 0";
  for (int n = 0; n < N; ++n)
    if (off[n + 1] < off[n]) return "R_offsets must be non-decreasing";
  if ((int64_t)P + off[N] > INT_MAX / 2) return "too many tokens";
  if ((int64_t)P + off[N] < 1) return "no tokens";
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return "Hq must be a positive multiple of Hkv";
  if (D != 64 && D != 128 && D != 512) return "D must be 64, 128 or 512";
  return nullptr;
}

void build_index(int P, int N, const int32_t* off, int32_t* seg_id, int32_t* pos_id, int32_t* cu_rep,
                 int32_t* rep2pack) {
  for (int t = 0; t < P; ++t) {
    if (seg_id) seg_id[t] = -1;
    if (pos_id) pos_id[t] = t;
  }
  for (int n = 0; n < N; ++n)
    for (int r = 0; r < off[n + 1] - off[n]; ++r) {
      const int t = P + off[n] + r;
      if (seg_id) seg_id[t] = n;
      if (pos_id) pos_id[t] = P + r;
    }
  int64_t x = 0;
  if (cu_rep) cu_rep[0] = 0;
  for (int n = 0; n < N; ++n) {
    const int len = P + off[n + 1] - off[n];
    for (int p = 0; p < len; ++p, ++x)
      if (rep2pack) rep2pack[x] = p < P ? p : P + off[n] + (p - P);
    if (cu_rep) cu_rep[n + 1] = (int32_t)x;
  }
}

namespace {

struct Region {
  int32_t row0, pos0, count;
};

std::vector<Region> regions(const Layout& L) {
  std::vector<Region> r;
  r.push_back({0, 0, L.P});
  for (int n = 0; n < L.N; ++n) r.push_back({L.P + L.off[n], L.P, L.off[n + 1] - L.off[n]});
  return r;
}

// tiles of `kr` (size `tile`) holding a key that some query in positions
// [p_first, p_last] attends
KeyRegion clip_keys(const Region& kr, int p_first, int p_last, int window, int tile) {
  KeyRegion k{kr.row0, kr.pos0, kr.count, 0, 0};
  if (kr.count <= 0) return k;
  int64_t lo = kr.pos0;
  if (window > 0) lo = std::max<int64_t>(lo, (int64_t)p_first - window + 1);
  const int64_t hi = std::min<int64_t>((int64_t)kr.pos0 + kr.count - 1, p_last);
  if (lo > hi) return k;
  k.t_lo = (int32_t)((lo - kr.pos0) / tile);
  k.t_hi = (int32_t)((hi - kr.pos0) / tile + 1);
  return k;
}

}  // namespace

std::vector<QTileItem> plan_qtiles(const Layout& L, int tile_rows, int key_tile) {
  std::vector<QTileItem> items;
  const auto regs = regions(L);
  for (size_t qr = 0; qr < regs.size(); ++qr) {
    const Region& q = regs[qr];
    for (int a = 0; a < q.count; a += tile_rows) {
      QTileItem it{};
      it.q_row0 = q.row0 + a;
      it.q_pos0 = q.pos0 + a;
      it.q_rows = std::min(tile_rows, q.count - a);
      const int p_first = it.q_pos0, p_last = it.q_pos0 + it.q_rows - 1;
      it.reg[0] = clip_keys(regs[0], p_first, p_last, L.window, key_tile);
      if (qr == 0)
        it.reg[1] = KeyRegion{q.row0, q.pos0, 0, 0, 0};  // prompt queries: one region
      else
        it.reg[1] = clip_keys(q, p_first, p_last, L.window, key_tile);
      const int gs = L.Hq / L.Hkv;
      for (int h = L.kv_begin() * gs; h < L.kv_end() * gs; ++h) {
        it.head = h;
        items.push_back(it);
      }
    }
  }
  std::stable_sort(items.begin(), items.end(), [](const QTileItem& a, const QTileItem& b) {
    const int ca = (a.reg[0].t_hi - a.reg[0].t_lo) + (a.reg[1].t_hi - a.reg[1].t_lo);
    const int cb = (b.reg[0].t_hi - b.reg[0].t_lo) + (b.reg[1].t_hi - b.reg[1].t_lo);
    return ca > cb;
  });
  return items;
}

KVPlan plan_kvtiles(const Layout& L, int key_tile, int q_block, int max_iters) {
  KVPlan plan;
  const auto regs = regions(L);
  const int gs = L.Hq / L.Hkv;
  struct TileList {
    int32_t k_row0, k_pos0, k_rows, begin, len;
  };
  std::vector<TileList> tiles;
  for (size_t kr = 0; kr < regs.size(); ++kr) {
    const Region& k = regs[kr];
    for (int a = 0; a < k.count; a += key_tile) {
      TileList tl{k.row0 + a, k.pos0 + a, std::min(key_tile, k.count - a), (int32_t)plan.qblocks.size(), 0};
      const int kp_first = tl.k_pos0, kp_last = tl.k_pos0 + tl.k_rows - 1;
      // query regions that see region kr: its own for a segment; for the prompt, every
      // segment (0..N-1) first and then the prompt itself, so that the long common part
      // of all prompt key tiles' walks comes first and lines up across tiles (L2 reuse)
      std::vector<size_t> qorder;
      if (kr == 0) {
        for (size_t qr = 1; qr < regs.size(); ++qr) qorder.push_back(qr);
        qorder.push_back(0);
      } else {
        qorder.push_back(kr);
      }
      for (size_t qr : qorder) {
        const Region& q = regs[qr];
        if (q.count <= 0) continue;
        int64_t lo = std::max<int64_t>(kp_first, q.pos0);
        int64_t hi = (int64_t)q.pos0 + q.count - 1;
        if (L.window > 0) hi = std::min<int64_t>(hi, (int64_t)kp_last + L.window - 1);
        if (lo > hi) continue;
        const int b_lo = (int)((lo - q.pos0) / q_block), b_hi = (int)((hi - q.pos0) / q_block + 1);
        for (int b = b_lo; b < b_hi; ++b)
          plan.qblocks.push_back(QBlock{q.row0 + b * q_block, q.pos0 + b * q_block, std::min(q_block, q.count - b * q_block)});
      }
      tl.len = (int32_t)plan.qblocks.size() - tl.begin;
      tiles.push_back(tl);
    }
  }
  // Chunks are emitted split-major (chunk s of every key tile of a kv-head, then
  // chunk s+1): CTAs that run together then stream the same query blocks.
  for (int g = L.kv_begin(); g < L.kv_end(); ++g) {
    std::vector<std::vector<KVTileItem>> per_tile;
    int max_split = 0;
    for (const TileList& tl : tiles) {
      const int total = gs * tl.len;
      const int nsplit = std::max(1, (total + max_iters - 1) / max_iters);
      const int chunk = (total + nsplit - 1) / nsplit;
      const int slot0 = plan.nslots;
      std::vector<KVTileItem> mine;
      for (int lo = 0; lo < total; lo += chunk) {
        KVTileItem it{};
        it.k_row0 = tl.k_row0;
        it.k_pos0 = tl.k_pos0;
        it.k_rows = tl.k_rows;
        it.kv_head = g;
        it.list_begin = tl.begin;
        it.list_len = tl.len;
        it.it_lo = lo;
        it.it_hi = std::min(total, lo + chunk);
        it.partial_slot = nsplit > 1 ? plan.nslots++ : -1;
        mine.push_back(it);
      }
      if (nsplit > 1) plan.reduces.push_back(ReduceItem{tl.k_row0, tl.k_rows, g, slot0, (int)mine.size(), 0});
      max_split = std::max(max_split, (int)mine.size());
      per_tile.push_back(std::move(mine));
    }
    for (int sidx = 0; sidx < max_split; ++sidx)
      for (const auto& mine : per_tile)
        if (sidx < (int)mine.size()) plan.items.push_back(mine[sidx]);
  }
  // heaviest first, on a coarse cost bucket so that equal-sized chunks keep their split-major order
  std::stable_sort(plan.items.begin(), plan.items.end(), [](const KVTileItem& a, const KVTileItem& b) {
    return (a.it_hi - a.it_lo) / 64 > (b.it_hi - b.it_lo) / 64;
  });
  return plan;
}

Plan512 plan_512(const Layout& L, const std::vector<QTileItem>& qitems, int max_iters) {
  Plan512 pl;
  const int gs = L.Hq / L.Hkv;
  constexpr int kTile = 128;
  // key tiles: prompt tiles first, then each segment's tiles
  std::vector<int32_t> seg_tile_base(L.N + 1, 0);
  const int prompt_tiles = (L.P + kTile - 1) / kTile;
  int ntiles = prompt_tiles;
  for (int n = 0; n < L.N; ++n) {
    seg_tile_base[n] = ntiles;
    ntiles += (L.off[n + 1] - L.off[n] + kTile - 1) / kTile;
  }
  pl.block_base.resize(qitems.size());
  int64_t nb = 0;
  for (size_t i = 0; i < qitems.size(); ++i) {
    pl.block_base[i] = (int32_t)nb;
    nb += (qitems[i].reg[0].t_hi - qitems[i].reg[0].t_lo) + (qitems[i].reg[1].t_hi - qitems[i].reg[1].t_lo);
  }
  pl.n_blocks = nb;
  // the segment whose rows begin at `row0` (and hold at least one row)
  auto seg_of_row = [&](int32_t row0) {
    for (int n = 0; n < L.N; ++n)
      if (L.P + L.off[n] == row0 && L.off[n + 1] > L.off[n]) return n;
    return -1;
  };
  // walk the query tiles in fixed order: group heads ascending, then packed row order
  std::vector<size_t> order(qitems.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
    if (qitems[a].head != qitems[b].head) return qitems[a].head < qitems[b].head;
    return qitems[a].q_row0 < qitems[b].q_row0;
  });
  std::vector<std::vector<XTEntry>> lists((size_t)ntiles * L.Hkv);
  for (size_t oi : order) {
    const QTileItem& it = qitems[oi];
    const int g = it.head / gs;
    int j = 0;
    for (int r = 0; r < 2; ++r) {
      const KeyRegion& kr = it.reg[r];
      const int base = r == 0 ? 0 : (kr.t_hi > kr.t_lo ? seg_tile_base[seg_of_row(kr.row0)] : 0);
      for (int t = kr.t_lo; t < kr.t_hi; ++t, ++j) {
        auto& lst = lists[(size_t)(base + t) * L.Hkv + g];
        for (int sub = 0; sub < 2; ++sub)
          if (sub * 64 < it.q_rows) lst.push_back(XTEntry{it.head, it.q_row0 + sub * 64, pl.block_base[oi] + j, sub});
      }
    }
  }
  // key tile geometry in the same numbering
  std::vector<std::pair<int32_t, int32_t>> ktile(ntiles);  // (row0, rows)
  for (int t = 0; t < prompt_tiles; ++t) ktile[t] = {t * kTile, std::min(kTile, L.P - t * kTile)};
  for (int n = 0; n < L.N; ++n) {
    const int R = L.off[n + 1] - L.off[n];
    for (int t = 0; t * kTile < R; ++t) ktile[seg_tile_base[n] + t] = {L.P + L.off[n] + t * kTile, std::min(kTile, R - t * kTile)};
  }
  for (int g = L.kv_begin(); g < L.kv_end(); ++g)
    for (int kt = 0; kt < ntiles; ++kt) {
      const auto& lst = lists[(size_t)kt * L.Hkv + g];
      const int begin = (int)pl.entries.size();
      pl.entries.insert(pl.entries.end(), lst.begin(), lst.end());
      const int total = (int)lst.size();
      const int nsplit = std::max(1, (total + max_iters - 1) / max_iters);
      const int chunk = std::max(1, (total + nsplit - 1) / nsplit);
      const int slot0 = pl.nslots;
      int made = 0;
      for (int lo = 0; lo < std::max(total, 1); lo += chunk, ++made) {
        XTItem x{};
        x.k_row0 = ktile[kt].first;
        x.k_rows = ktile[kt].second;
        x.kv_head = g;
        x.list_begin = begin;
        x.it_lo = lo;
        x.it_hi = std::min(total, lo + chunk);
        x.partial_slot = nsplit > 1 ? pl.nslots++ : -1;
        pl.items.push_back(x);
      }
      if (nsplit > 1) pl.reduces.push_back(ReduceItem{ktile[kt].first, ktile[kt].second, g, slot0, made, 0});
    }
  std::stable_sort(pl.items.begin(), pl.items.end(),
                   [](const XTItem& a, const XTItem& b) { return (a.it_hi - a.it_lo) > (b.it_hi - b.it_lo); });
  return pl;
}

}  // namespace dkv
