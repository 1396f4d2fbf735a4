// Host side of the C ABI: descriptor validation, the largest-first work queues, plans,
// workspace layout and the dispatch of the compute calls to their kernels.
//
// AugTree, "Splitting Prompt Prefill from Response Replay for Context-Parallel
// Long-Context LLM Post-Training":
//   Sec. 3.1        replay tree T = (P, {R_i}) per group (the ragged descriptors);
//   Sec. 3.2        prefill once, replay many; Eq. 1 valid KV context; Eq. 2 prompt
//                   K/V gradient summed over all branches;
//   Sec. 3.4        bounded replay units with work weights, largest-first greedy
//                   balancing (the work queues built here; thread blocks are the lanes).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <tuple>
#include <utility>

#include "internal.h"

using namespace augtree;

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Grp {
  int64_t p0, lp, r0, lr;
  std::vector<int64_t> starts, ends;  // branch row ranges (global response rows)
};

bool read_groups(const std::vector<int32_t>& po, const std::vector<int32_t>& bb,
                 const std::vector<int32_t>& ro, std::vector<Grp>& out) {
  const int ng = (int)po.size() - 1;
  out.resize(ng);
  for (int g = 0; g < ng; ++g) {
    Grp& G = out[g];
    G.p0 = po[g];
    G.lp = (int64_t)po[g + 1] - po[g];
    G.r0 = ro[bb[g]];
    G.lr = (int64_t)ro[bb[g + 1]] - ro[bb[g]];
    for (int b = bb[g]; b < bb[g + 1]; ++b) {
      G.starts.push_back(ro[b]);
      G.ends.push_back(ro[b + 1]);
    }
  }
  return true;
}

// Index (within the group) of the non-empty branch holding global response row `row`.
int branch_of(const Grp& G, int64_t row) {
  auto it = std::upper_bound(G.starts.begin(), G.starts.end(), row);
  int i = (int)(it - G.starts.begin()) - 1;
  while (i >= 0 && !(G.starts[i] <= row && row < G.ends[i])) --i;  // skip empty branches
  return i;
}

struct Item {
  int32_t w[AUGTREE_ITEM_WORDS];
};

augtree_status validate_desc(const augtree_desc* d, std::vector<int32_t>& po, std::vector<int32_t>& bb,
                             std::vector<int32_t>& ro) {
  if (!d || !d->prompt_off || !d->branch_begin || !d->resp_off) return AUGTREE_ERR_INVALID_ARG;
  if (d->n_groups < 0 || d->n_branches < 0) return AUGTREE_ERR_INVALID_ARG;
  po.assign(d->prompt_off, d->prompt_off + d->n_groups + 1);
  bb.assign(d->branch_begin, d->branch_begin + d->n_groups + 1);
  ro.assign(d->resp_off, d->resp_off + d->n_branches + 1);
  if (po[0] != 0 || bb[0] != 0 || ro[0] != 0) return AUGTREE_ERR_INVALID_ARG;
  if (bb[d->n_groups] != d->n_branches) return AUGTREE_ERR_INVALID_ARG;
  for (int g = 0; g < d->n_groups; ++g)
    if (po[g + 1] < po[g] || bb[g + 1] < bb[g]) return AUGTREE_ERR_INVALID_ARG;
  for (int b = 0; b < d->n_branches; ++b)
    if (ro[b + 1] < ro[b]) return AUGTREE_ERR_INVALID_ARG;
  return AUGTREE_OK;
}

augtree_status validate_cfg(const augtree_config* c, bool need_sms) {
  if (!c) return AUGTREE_ERR_INVALID_ARG;
  if (c->hq <= 0 || c->hkv <= 0) return AUGTREE_ERR_INVALID_ARG;
  if (c->schedule != AUGTREE_SCHED_QUEUE && c->schedule != AUGTREE_SCHED_PERSISTENT) return AUGTREE_ERR_INVALID_ARG;
  if (c->num_sms < 0 || (need_sms && c->num_sms == 0)) return AUGTREE_ERR_INVALID_ARG;
  if (!(c->softmax_scale >= 0.0f) || std::isinf(c->softmax_scale)) return AUGTREE_ERR_INVALID_ARG;
  if (c->hq % c->hkv != 0) return AUGTREE_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return AUGTREE_ERR_UNSUPPORTED;
  if (c->dtype != AUGTREE_FP32 && c->dtype != AUGTREE_BF16) return AUGTREE_ERR_UNSUPPORTED;
  if (c->kernel < AUGTREE_KERNEL_AUTO || c->kernel > AUGTREE_KERNEL_TC) return AUGTREE_ERR_INVALID_ARG;
  if (c->kernel == AUGTREE_KERNEL_TC && (c->dtype != AUGTREE_BF16 || c->head_dim != 128))
    return AUGTREE_ERR_UNSUPPORTED;
  return AUGTREE_OK;
}

int resolve_family(const augtree_config* c) {
  if (c->kernel == AUGTREE_KERNEL_SIMT) return AUGTREE_KERNEL_SIMT;
  if (c->kernel == AUGTREE_KERNEL_TC) return AUGTREE_KERNEL_TC;
  return (c->dtype == AUGTREE_BF16 && c->head_dim == 128) ? AUGTREE_KERNEL_TC : AUGTREE_KERNEL_SIMT;
}

void tiles_for(int family, int op, int* bm, int* bn) {
  if (family == AUGTREE_KERNEL_TC) {
    // 128 keys per KV tile; 128 query rows per query tile (the backward's key-side
    // queue walks tiles of kTcBwdKvRows rows).
    *bn = 128;
    *bm = (op == AUGTREE_OP_PREFILL_FWD || op == AUGTREE_OP_REPLAY_FWD) ? 128 : kTcBwdKvRows;
  } else {
    *bm = 64;
    *bn = 64;
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

namespace augtree {

namespace {
// Splits of a replay query tile walking c KV tiles at about T tiles per split.
int64_t fwd_split_count(int64_t c, int64_t T) {
  const int64_t s = std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, cdiv(c, T)));
  return c > 0 ? cdiv(c, cdiv(c, s)) : 1;
}
}  // namespace

void replay_fwd_splits(const std::vector<int64_t>& costs, int hq, int hkv, int num_sms, std::vector<int64_t>& splits) {
  // Split-KV of the replay forward (Sec. 3.3: partial states over disjoint key ranges
  // merge exactly).  Only a queue with fewer than 2 * num_sms items (too few blocks for
  // the GPU) is split.  The chunk T is the one of the candidates ceil(c_max / s),
  // s = 1..64 (c_max the largest tile cost, T >= kFwdMinChunk for s > 1, at most
  // kMaxFwdParts partial states) that minimises the estimated time
  //   ceil(blocks / num_sms) * (largest chunk + kFwdBlockOverhead)
  // (waves of blocks times the longest block; a block is one split of a tile for one
  // query head); ties keep the larger T.
  (void)hkv;
  splits.assign(costs.size(), 1);
  const int64_t n_items = (int64_t)costs.size() * hq;
  if (n_items == 0 || n_items >= 2 * (int64_t)num_sms) return;
  const int64_t per_tile = hq;
  int64_t cmax = 0;
  for (int64_t c : costs) cmax = std::max(cmax, c);
  int64_t best_t = cmax, best_time = -1;
  for (int64_t sc = 1; sc <= kMaxSplit; ++sc) {
    const int64_t T = cdiv(cmax, sc);
    if (sc > 1 && T < kFwdMinChunk) break;
    int64_t blocks = 0, parts = 0, chunk_max = 0;
    for (int64_t c : costs) {
      const int64_t st = fwd_split_count(c, T);
      blocks += per_tile * st;
      if (st > 1) parts += (int64_t)hq * st;
      chunk_max = std::max(chunk_max, cdiv(c, st));
    }
    if (parts > kMaxFwdParts) continue;
    const int64_t time = cdiv(blocks, num_sms) * (chunk_max + kFwdBlockOverhead);
    if (best_time < 0 || time < best_time) {
      best_time = time;
      best_t = T;
    }
  }
  for (size_t i = 0; i < costs.size(); ++i) splits[i] = fwd_split_count(costs[i], best_t);
}

augtree_status build_queue(const std::vector<int32_t>& po, const std::vector<int32_t>& bb,
                           const std::vector<int32_t>& ro, int hq, int hkv, int op, int bm, int bn,
                           int num_sms, bool split_fwd, std::vector<int32_t>& out) {
  std::vector<Grp> groups;
  read_groups(po, bb, ro, groups);
  const int r = hq / hkv;
  std::vector<Item> items;
  // Key-side queues: the branch (index within the group) whose query tiles a response-key
  // item walks, -1 for prompt-key items (they walk the group's query tiles).
  std::vector<int32_t> walk_branch;
  // Replay forward queue: the branch of the query tile's first row, whose keys the item's
  // own-branch tiles are (-1 elsewhere).
  std::vector<int32_t> row_branch;
  auto push = [&](int kind, int g, int64_t tile, int head, int split, int64_t cost, int64_t a, int64_t b,
                  int branch = -1, int rbranch = -1) {
    Item it;
    it.w[0] = kind; it.w[1] = g; it.w[2] = (int32_t)tile; it.w[3] = head;
    it.w[4] = split; it.w[5] = (int32_t)cost; it.w[6] = (int32_t)a; it.w[7] = (int32_t)b;
    items.push_back(it);
    walk_branch.push_back(branch);
    row_branch.push_back(rbranch);
  };
  const int ng = (int)groups.size();
  if (op == AUGTREE_OP_PREFILL_FWD) {
    for (int g = 0; g < ng; ++g) {
      const Grp& G = groups[g];
      for (int64_t t = 0; t < cdiv(G.lp, bm); ++t) {
        int64_t row_end = std::min(G.p0 + (t + 1) * bm, G.p0 + G.lp);
        int64_t a = cdiv(row_end - G.p0, bn);
        for (int h = 0; h < hq; ++h) push(K_PREFILL_Q, g, t, h, 0, a, a, 0);
      }
    }
  } else if (op == AUGTREE_OP_REPLAY_FWD) {
    struct RT { int g; int64_t t, a, b; int br; };
    std::vector<RT> tiles;
    std::vector<int64_t> costs;
    for (int g = 0; g < ng; ++g) {
      const Grp& G = groups[g];
      int64_t a = cdiv(G.lp, bn);
      for (int64_t t = 0; t < cdiv(G.lr, bm); ++t) {
        int64_t row_begin = G.r0 + t * bm;
        int64_t row_end = std::min(row_begin + bm, G.r0 + G.lr);
        const int br = branch_of(G, row_begin);
        int64_t bstart = G.starts[br];
        int64_t b = cdiv(row_end - bstart, bn);
        tiles.push_back({g, t, a, b, br});
        costs.push_back(a + b);
      }
    }
    std::vector<int64_t> splits(tiles.size(), 1);
    if (split_fwd) replay_fwd_splits(costs, hq, hkv, num_sms, splits);
    for (size_t i = 0; i < tiles.size(); ++i) {
      const RT& x = tiles[i];
      const int64_t cost = x.a + x.b, s = splits[i], c = cdiv(cost, s);
      for (int64_t k = 0; k < s; ++k) {
        const int64_t kc = s == 1 ? cost : std::min(c, cost - k * c);
        for (int h = 0; h < hq; ++h) push(K_REPLAY_Q, x.g, x.t, h, (int)k, kc, x.a, x.b, -1, x.br);
      }
    }
  } else if (op == AUGTREE_OP_REPLAY_BWD || op == AUGTREE_OP_TREE_BWD) {
    // Costs before splitting fix the split target (replay items only, in both queues).
    const bool tree = op == AUGTREE_OP_TREE_BWD;
    int64_t total = 0;
    struct RI { int g; int64_t j, qa, qb; int br; };
    std::vector<RI> resp;
    for (int g = 0; g < ng; ++g) {
      const Grp& G = groups[g];
      int64_t nq = cdiv(G.lr, bm);
      int64_t nkp = nq > 0 ? cdiv(G.lp, bn) : 0;
      total += nkp * nq * r * hkv;
      for (int64_t j = 0; j < cdiv(G.lr, bn); ++j) {
        int64_t k_lo = G.r0 + j * bn;
        int64_t k_hi = std::min(k_lo + bn, G.r0 + G.lr);
        int64_t e = G.ends[branch_of(G, k_hi - 1)];
        int64_t qa = (k_lo - G.r0) / bm;
        int64_t qb = cdiv(e - G.r0, bm);
        resp.push_back({g, j, qa, qb, branch_of(G, k_lo)});
        total += (qb - qa) * r * hkv;
      }
    }
    int64_t target = std::max<int64_t>(r, cdiv(total, 2 * (int64_t)num_sms));
    for (int g = 0; g < ng; ++g) {
      const Grp& G = groups[g];
      int64_t nq = cdiv(G.lr, bm);
      const int64_t nqp = cdiv(G.lp, bm);
      if (G.lp == 0 || (nq == 0 && !tree)) continue;
      if (nq == 0) {
        // Fused backward, no response rows: the prompt's own causal part only.
        for (int64_t j = 0; j < cdiv(G.lp, bn); ++j)
          for (int h = 0; h < hkv; ++h) push(K_TREE_PROMPT_KV, g, j, h, 0, (nqp - (j * bn) / bm) * r, 0, 0);
        continue;
      }
      int64_t s = std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, cdiv(nq * r, target)));
      int64_t c = cdiv(nq, s);
      s = cdiv(nq, c);
      for (int64_t j = 0; j < cdiv(G.lp, bn); ++j)
        for (int64_t k = 0; k < s; ++k) {
          int64_t qa = k * c, qb = std::min((k + 1) * c, nq);
          // In the fused backward, split 0 also walks the prompt's own causal query
          // tiles of this KV tile.
          const int64_t own = (tree && k == 0) ? nqp - (j * bn) / bm : 0;
          for (int h = 0; h < hkv; ++h)
            push(tree ? K_TREE_PROMPT_KV : K_PROMPT_KV, g, j, h, (int)k, (qb - qa + own) * r, qa, qb);
        }
    }
    for (const RI& x : resp)
      for (int h = 0; h < hkv; ++h) push(K_RESP_KV, x.g, x.j, h, 0, (x.qb - x.qa) * r, x.qa, x.qb, x.br);
  } else if (op == AUGTREE_OP_PREFILL_BWD) {
    for (int g = 0; g < ng; ++g) {
      const Grp& G = groups[g];
      int64_t nq = cdiv(G.lp, bm);
      for (int64_t j = 0; j < cdiv(G.lp, bn); ++j) {
        int64_t qa = (j * bn) / bm;
        for (int h = 0; h < hkv; ++h) push(K_PREFILL_KV, g, j, h, 0, (nq - qa) * r, qa, nq);
      }
    }
  } else {
    return AUGTREE_ERR_INVALID_ARG;
  }
  // Every item walks the K/V or Q/dO tiles of one stream: a forward item the K/V of its
  // group's KV head, a key-side item the query tiles of its group for its KV head or,
  // for response keys, of one branch.  Items of one stream form a chunk; chunks run
  // largest first (by total cost; ties by group, KV head, branch with -1 for a
  // group-wide stream).  Within a chunk, replay forward items form sub-chunks by the
  // branch of their query tile's first row (whose own-branch K/V they read), largest
  // first (ties by branch); every other item is its chunk's only sub-chunk.  Items
  // within a sub-chunk run largest first (ties by tile, kind, split, head).  Blocks that
  // run side by side then mostly share one stream, which L2 holds once for all of them;
  // the queues stay balanced (largest first within sub-chunks).
  const bool fwd = op == AUGTREE_OP_PREFILL_FWD || op == AUGTREE_OP_REPLAY_FWD;
  using CKey = std::tuple<int32_t, int32_t, int32_t>;
  using SKey = std::tuple<int32_t, int32_t, int32_t, int32_t>;
  auto chunk_of = [&](size_t i) {
    return CKey(items[i].w[1], fwd ? items[i].w[3] / r : items[i].w[3], walk_branch[i]);
  };
  auto sub_of = [&](size_t i) {
    const CKey c = chunk_of(i);
    return SKey(std::get<0>(c), std::get<1>(c), std::get<2>(c), row_branch[i]);
  };
  // Total cost per key, looked up by binary search in a sorted table.
  auto totals_of = [&](auto key_of) {
    using K = decltype(key_of(size_t(0)));
    std::vector<std::pair<K, int64_t>> cs(items.size()), tot;
    for (size_t i = 0; i < items.size(); ++i) cs[i] = {key_of(i), (int64_t)items[i].w[5]};
    std::sort(cs.begin(), cs.end());
    for (size_t i = 0; i < cs.size();) {
      size_t k = i;
      int64_t t = 0;
      while (k < cs.size() && cs[k].first == cs[i].first) t += cs[k++].second;
      tot.push_back({cs[i].first, t});
      i = k;
    }
    return tot;
  };
  const auto chunk_tot = totals_of(chunk_of);
  const auto sub_tot = totals_of(sub_of);
  auto lookup = [](const auto& tab, const auto& key) {
    auto pos = std::lower_bound(tab.begin(), tab.end(), key,
                                [](const auto& e, const auto& v) { return e.first < v; });
    return pos->second;
  };
  struct Key {
    int64_t chunk_cost, sub_cost;
    int32_t g, h, br, sb;
    size_t idx;
  };
  std::vector<Key> keys(items.size());
  for (size_t i = 0; i < items.size(); ++i) {
    const CKey c = chunk_of(i);
    keys[i] = Key{lookup(chunk_tot, c), lookup(sub_tot, sub_of(i)), std::get<0>(c), std::get<1>(c), std::get<2>(c),
                  row_branch[i], i};
  }
  std::sort(keys.begin(), keys.end(), [&](const Key& x, const Key& y) {
    if (x.chunk_cost != y.chunk_cost) return x.chunk_cost > y.chunk_cost;
    if (x.g != y.g) return x.g < y.g;
    if (x.h != y.h) return x.h < y.h;
    if (x.br != y.br) return x.br < y.br;
    if (x.sub_cost != y.sub_cost) return x.sub_cost > y.sub_cost;
    if (x.sb != y.sb) return x.sb < y.sb;
    const Item& a = items[x.idx];
    const Item& b = items[y.idx];
    if (a.w[5] != b.w[5]) return a.w[5] > b.w[5];
    if (a.w[2] != b.w[2]) return a.w[2] < b.w[2];
    if (a.w[0] != b.w[0]) return a.w[0] < b.w[0];
    if (a.w[4] != b.w[4]) return a.w[4] < b.w[4];
    return a.w[3] < b.w[3];
  });
  std::vector<Item> sorted(items.size());
  for (size_t i = 0; i < keys.size(); ++i) sorted[i] = items[keys[i].idx];
  items.swap(sorted);
  out.resize(items.size() * AUGTREE_ITEM_WORDS);
  if (!items.empty()) std::memcpy(out.data(), items.data(), items.size() * sizeof(Item));
  return AUGTREE_OK;
}

augtree_status build_lanes(const std::vector<int32_t>& q, int unit_items, int lanes, LaneSet& out) {
  out.off.clear();
  out.units.clear();
  const int64_t n_units = (int64_t)(q.size() / AUGTREE_ITEM_WORDS) / unit_items;
  if (n_units > INT32_MAX || lanes < 1) return AUGTREE_ERR_INVALID_ARG;
  const int L = (int)std::min<int64_t>(lanes, n_units);
  out.n_lanes = L;
  out.off.assign((size_t)L + 1, 0);
  if (n_units == 0) return AUGTREE_OK;
  // Unit weight: its items' cost (the items of a unit share one tile, hence one cost).
  std::vector<int64_t> w((size_t)n_units);
  for (int64_t u = 0; u < n_units; ++u) w[u] = (int64_t)q[(size_t)u * unit_items * AUGTREE_ITEM_WORDS + 5] * unit_items;
  const int rounds = (int)((n_units + L - 1) / L);
  std::vector<int32_t> rnd((size_t)n_units), lane((size_t)n_units);
  int64_t makespan = 0;
  augtree_status st = augtree_assign_grid(w.data(), (int32_t)n_units, rounds, L, AUGTREE_LANES_EXACT_UNITS,
                                          rnd.data(), lane.data(), &makespan, nullptr);
  if (st != AUGTREE_OK) return st;
  for (int64_t u = 0; u < n_units; ++u) out.off[lane[u] + 1] += 1;
  for (int l = 0; l < L; ++l) out.off[l + 1] += out.off[l];
  out.units.assign((size_t)n_units, 0);
  for (int64_t u = 0; u < n_units; ++u) out.units[out.off[lane[u]] + rnd[u]] = (int32_t)u;
  return AUGTREE_OK;
}

// Row statistics of the backward: SIMT kernels read Delta [Hq, rows]; tensor-core
// kernels read tiles of {lse * log2(e), Delta} [Hq, tiles, 2 x 64] (one bulk copy each).
static size_t stats_bytes(const augtree_plan* p, bool prompt_side) {
  const size_t hq = p->cfg.hq;
  if (p->family == AUGTREE_KERNEL_TC)
    return hq * (size_t)(prompt_side ? p->ntiles_p : p->ntiles_r) * 2 * kStatRows * 4;
  return hq * (size_t)(prompt_side ? p->total_prompt : p->total_resp) * 4;
}

// The tensor-core backward writes dQ once per query tile (no fp32 accumulator).
static size_t dq_acc_bytes(const augtree_plan* p, size_t rows) {
  return p->family == AUGTREE_KERNEL_TC ? 0 : align256(rows * p->cfg.hq * p->cfg.head_dim * 4);
}

// Tensor-core family: the key-side kernel's {-lse/s, -Delta} rows per query tile.
static size_t aug_bytes(const augtree_plan* p, bool prompt_side) {
  if (p->family != AUGTREE_KERNEL_TC) return 0;
  return align256((size_t)p->cfg.hq * (prompt_side ? p->ntiles_p : p->ntiles_r) * kAugTileBytes);
}

FwdWorkspace replay_fwd_ws(const augtree_plan* p) {
  FwdWorkspace w;
  const size_t n = (size_t)p->n_fwd_parts;
  w.o_off = 0;
  w.lse_off = align256(n * kFwdPartRows * p->cfg.head_dim * 4);
  w.total = n ? w.lse_off + align256(n * kFwdPartRows * 4) : 0;
  return w;
}

BwdWorkspace replay_bwd_ws(const augtree_plan* p) {
  BwdWorkspace w;
  const size_t hkv = p->cfg.hkv, d = p->cfg.head_dim, R = p->total_resp;
  w.delta_off = 0;
  w.aug_off = align256(stats_bytes(p, false));
  w.dq_off = w.aug_off + aug_bytes(p, false);
  w.dkpart_off = w.dq_off + dq_acc_bytes(p, R);
  w.dvpart_off = w.dkpart_off + align256((size_t)p->part_rows * hkv * d * 4);
  w.dqpart_off = w.dvpart_off + align256((size_t)p->part_rows * hkv * d * 4);
  w.slots_off = w.dqpart_off + align256((size_t)p->n_fwd_parts * kFwdPartRows * d * 4);
  w.total = w.slots_off + (p->family == AUGTREE_KERNEL_TC ? kFlushSlots * kFlushSlotBytes : 0);
  return w;
}

TreeWorkspace tree_bwd_ws(const augtree_plan* p) {
  TreeWorkspace t;
  t.r = replay_bwd_ws(p);
  t.p = prefill_bwd_ws(p);
  // The replay part keeps its flush slots; the prefill part needs none of its own (the
  // kernels run one after the other).
  t.p_off = align256(t.r.total);
  t.sum_off = align256(t.p_off + t.p.slots_off);
  const size_t sum_bytes =
      p->family == AUGTREE_KERNEL_TC ? 0 : align256((size_t)p->total_prompt * p->cfg.hkv * p->cfg.head_dim * 4);
  t.total = t.sum_off + 2 * sum_bytes;
  t.sum_bytes = sum_bytes;
  return t;
}

BwdWorkspace prefill_bwd_ws(const augtree_plan* p) {
  BwdWorkspace w;
  const size_t P = p->total_prompt;
  w.delta_off = 0;
  w.aug_off = align256(stats_bytes(p, true));
  w.dq_off = w.aug_off + aug_bytes(p, true);
  w.dkpart_off = w.dvpart_off = w.dqpart_off = w.slots_off = w.dq_off + dq_acc_bytes(p, P);
  w.total = w.slots_off + (p->family == AUGTREE_KERNEL_TC ? kFlushSlots * kFlushSlotBytes : 0);
  return w;
}

Geometry geometry(const augtree_plan* p) {
  Geometry g;
  g.groups = p->groups_d;
  g.row_bstart = p->row_bstart_d;
  g.splits = p->splits_d;
  g.fsplit = p->fsplit_d;
  g.hq = p->cfg.hq;
  g.hkv = p->cfg.hkv;
  g.d = p->cfg.head_dim;
  g.total_prompt = p->total_prompt;
  g.total_resp = p->total_resp;
  g.n_groups = p->n_groups;
  g.scale = p->cfg.softmax_scale > 0.f ? p->cfg.softmax_scale : 1.0f / std::sqrt((float)p->cfg.head_dim);
  g.scale_log2 = g.scale * 1.4426950408889634f;
  return g;
}

CallTimer::CallTimer(const augtree_plan* p, int op, cudaStream_t s) : p_(p), op_(op), slot_(0), n_(0), s_(s) {
  if (p_->timing.on) slot_ = (int)(p_->timing.calls[op_] % AUGTREE_TIMING_RING);
}
void CallTimer::mark(int kind) {
  auto& T = p_->timing;
  if (!T.on || n_ >= augtree_plan::kTimingMarks - 1) return;
  cudaEventRecord(T.ev[op_][slot_][n_], s_);
  T.kind[op_][slot_][n_] = kind;
  ++n_;
}
void CallTimer::finish() {
  auto& T = p_->timing;
  if (!T.on || n_ == 0) return;
  cudaEventRecord(T.ev[op_][slot_][n_], s_);
  T.n_marks[op_][slot_] = n_ + 1;
  T.calls[op_] += 1;
}

}  // namespace augtree

// =====================================================================================
// C ABI
// =====================================================================================
extern "C" {

const char* augtree_status_string(augtree_status s) {
  switch (s) {
    case AUGTREE_OK: return "ok";
    case AUGTREE_ERR_INVALID_ARG: return "invalid argument";
    case AUGTREE_ERR_UNSUPPORTED: return "unsupported configuration";
    case AUGTREE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case AUGTREE_ERR_CUDA: return "CUDA error";
    case AUGTREE_ERR_DEVICE_CHECK: return "device-side check failed";
    case AUGTREE_ERR_TIMEOUT: return "device-side wait timed out";
    case AUGTREE_ERR_CAPACITY: return "output capacity too small";
  }
  return "unknown status";
}

int32_t augtree_version(void) { return 200; }  // 0.2.0: augtree_tree_bwd, augtree_assign_grid

augtree_status augtree_tile_sizes(const augtree_config* cfg, int32_t op, int32_t* bm, int32_t* bn) {
  augtree_status st = validate_cfg(cfg, false);
  if (st != AUGTREE_OK) return st;
  if (!bm || !bn || op < 0 || op >= kNumOps) return AUGTREE_ERR_INVALID_ARG;
  int m, n;
  tiles_for(resolve_family(cfg), op, &m, &n);
  *bm = m;
  *bn = n;
  return AUGTREE_OK;
}

augtree_status augtree_schedule_build(const augtree_desc* desc, const augtree_config* cfg, int32_t op,
                                      int32_t* out, size_t cap_items, size_t* n_items) {
  std::vector<int32_t> po, bb, ro;
  augtree_status st = validate_desc(desc, po, bb, ro);
  if (st != AUGTREE_OK) return st;
  if ((st = validate_cfg(cfg, true)) != AUGTREE_OK) return st;
  if (!n_items || op < 0 || op >= kNumOps || (cap_items > 0 && !out)) return AUGTREE_ERR_INVALID_ARG;
  int bm, bn;
  tiles_for(resolve_family(cfg), op, &bm, &bn);
  std::vector<int32_t> q;
  try {
    st = build_queue(po, bb, ro, cfg->hq, cfg->hkv, op, bm, bn, cfg->num_sms,
                     resolve_family(cfg) == AUGTREE_KERNEL_TC, q);
  } catch (const std::bad_alloc&) {
    return AUGTREE_ERR_CAPACITY;
  }
  if (st != AUGTREE_OK) return st;
  *n_items = q.size() / AUGTREE_ITEM_WORDS;
  if (*n_items > cap_items) return AUGTREE_ERR_CAPACITY;
  if (!q.empty()) std::memcpy(out, q.data(), q.size() * sizeof(int32_t));
  return AUGTREE_OK;
}

augtree_status augtree_schedule_lanes(const augtree_desc* desc, const augtree_config* cfg, int32_t op,
                                      int32_t kernel_id, int32_t* lane_off, size_t cap_lanes, int32_t* units,
                                      size_t cap_units, size_t* n_lanes, size_t* n_units) {
  std::vector<int32_t> po, bb, ro;
  augtree_status st = validate_desc(desc, po, bb, ro);
  if (st != AUGTREE_OK) return st;
  if ((st = validate_cfg(cfg, true)) != AUGTREE_OK) return st;
  if (!n_lanes || !n_units || op < 0 || op >= kNumOps) return AUGTREE_ERR_INVALID_ARG;
  const bool fwd_op = op <= AUGTREE_OP_REPLAY_FWD;
  if (kernel_id != AUGTREE_KID_BWD_QUERY_SIDE && kernel_id != AUGTREE_KID_BWD_KEY_SIDE) return AUGTREE_ERR_INVALID_ARG;
  if ((kernel_id == AUGTREE_KID_BWD_QUERY_SIDE) != fwd_op) return AUGTREE_ERR_INVALID_ARG;
  int bm, bn;
  tiles_for(resolve_family(cfg), op, &bm, &bn);
  std::vector<int32_t> q;
  LaneSet l;
  try {
    st = build_queue(po, bb, ro, cfg->hq, cfg->hkv, op, bm, bn, cfg->num_sms,
                     resolve_family(cfg) == AUGTREE_KERNEL_TC, q);
    if (st != AUGTREE_OK) return st;
    st = build_lanes(q, 1, cfg->num_sms, l);
  } catch (const std::bad_alloc&) {
    return AUGTREE_ERR_CAPACITY;
  }
  if (st != AUGTREE_OK) return st;
  *n_lanes = (size_t)l.n_lanes;
  *n_units = l.units.size();
  if (*n_lanes + 1 > cap_lanes || *n_units > cap_units) return AUGTREE_ERR_CAPACITY;
  if (lane_off) std::memcpy(lane_off, l.off.data(), l.off.size() * sizeof(int32_t));
  if (units && !l.units.empty()) std::memcpy(units, l.units.data(), l.units.size() * sizeof(int32_t));
  return AUGTREE_OK;
}

augtree_status augtree_plan_destroy(augtree_plan* p) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != p->device) cudaSetDevice(p->device);
  cudaFree(p->groups_d);
  cudaFree(p->row_bstart_d);
  cudaFree(p->row_bend_d);
  cudaFree(p->splits_d);
  cudaFree(p->fsplit_d);
  cudaFree(p->fsplit_tiles_d);
  cudaFree(p->err_d);
  for (int i = 0; i < kNumOps; ++i) cudaFree(p->queue_d[i]);
  for (int i = 0; i < 2; ++i) {
    cudaFree(p->lanes_dq[i].off_d);
    cudaFree(p->lanes_dq[i].units_d);
  }
  for (int i = 0; i < kNumOps; ++i) {
    cudaFree(p->lanes_kv[i].off_d);
    cudaFree(p->lanes_kv[i].units_d);
  }
  if (p->timing.created)
    for (int op = 0; op < kNumOps; ++op)
      for (int c = 0; c < AUGTREE_TIMING_RING; ++c)
        for (int k = 0; k < augtree_plan::kTimingMarks; ++k) cudaEventDestroy(p->timing.ev[op][c][k]);
  if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
  delete p;
  return AUGTREE_OK;
}

augtree_status augtree_plan_create(const augtree_desc* desc, const augtree_config* cfg, augtree_plan** out) {
  if (!out) return AUGTREE_ERR_INVALID_ARG;
  *out = nullptr;
  std::vector<int32_t> po, bb, ro;
  augtree_status st = validate_desc(desc, po, bb, ro);
  if (st != AUGTREE_OK) return st;
  if ((st = validate_cfg(cfg, false)) != AUGTREE_OK) return st;
  augtree_plan* p = new (std::nothrow) augtree_plan();
  if (!p) return AUGTREE_ERR_CUDA;
  p->cfg = *cfg;
  p->groups_d = nullptr;
  p->err_d = nullptr;
  p->row_bstart_d = nullptr;
  p->row_bend_d = nullptr;
  p->splits_d = nullptr;
  p->fsplit_d = nullptr;
  p->fsplit_tiles_d = nullptr;
  p->n_fwd_parts = 0;
  p->static_scratch = nullptr;
  for (int i = 0; i < kNumOps; ++i) p->queue_d[i] = nullptr;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return AUGTREE_ERR_CUDA;
  }
  if (p->cfg.num_sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess || sms <= 0) {
      delete p;
      return AUGTREE_ERR_CUDA;
    }
    p->cfg.num_sms = sms;
  }
  p->family = resolve_family(cfg);
  p->n_groups = desc->n_groups;
  p->n_branches = desc->n_branches;
  p->total_prompt = po[desc->n_groups];
  p->total_resp = ro[desc->n_branches];
  std::vector<Grp> groups;
  read_groups(po, bb, ro, groups);
  p->groups_h.resize(p->n_groups);
  for (int g = 0; g < p->n_groups; ++g)
    p->groups_h[g] = GroupInfo{(int32_t)groups[g].p0, (int32_t)groups[g].lp, (int32_t)groups[g].r0,
                               (int32_t)groups[g].lr, 0, 0};
  p->ntiles_p = p->ntiles_r = 0;
  for (int g = 0; g < p->n_groups; ++g) {
    p->groups_h[g].tp0 = p->ntiles_p;
    p->groups_h[g].tr0 = p->ntiles_r;
    p->ntiles_p += (int32_t)cdiv(p->groups_h[g].lp, kStatRows);
    p->ntiles_r += (int32_t)cdiv(p->groups_h[g].lr, kStatRows);
  }
  std::vector<int32_t> bstart(std::max(1, p->total_resp)), bend(std::max(1, p->total_resp));
  for (int b = 0; b < p->n_branches; ++b)
    for (int32_t row = ro[b]; row < ro[b + 1]; ++row) {
      bstart[row] = ro[b];
      bend[row] = ro[b + 1];
    }
  for (int op = 0; op < kNumOps; ++op) {
    tiles_for(p->family, op, &p->bm[op], &p->bn[op]);
    st = build_queue(po, bb, ro, cfg->hq, cfg->hkv, op, p->bm[op], p->bn[op], p->cfg.num_sms,
                     p->family == AUGTREE_KERNEL_TC, p->queue_h[op]);
    if (st != AUGTREE_OK) {
      delete p;
      return st;
    }
    p->n_items[op] = p->queue_h[op].size() / AUGTREE_ITEM_WORDS;
  }
  // Persistent schedule: AssignGrid's placement of every tensor-core kernel's units.
  if (p->family == AUGTREE_KERNEL_TC && cfg->schedule == AUGTREE_SCHED_PERSISTENT) {
    for (int op = 0; op < kNumOps && st == AUGTREE_OK; ++op) {
      if (op <= AUGTREE_OP_REPLAY_FWD) {
        st = build_lanes(p->queue_h[op], 1, p->cfg.num_sms, p->lanes_dq[op]);
      } else {
        st = build_lanes(p->queue_h[op], 1, p->cfg.num_sms, p->lanes_kv[op]);
      }
    }
    if (st != AUGTREE_OK) {
      delete p;
      return st;
    }
  }
  // Split-K bookkeeping from the replay backward queue.
  p->splits_h.assign(std::max(1, p->n_groups), SplitInfo{0, 0, 0});
  for (size_t i = 0; i < p->n_items[AUGTREE_OP_REPLAY_BWD]; ++i) {
    const int32_t* it = &p->queue_h[AUGTREE_OP_REPLAY_BWD][i * AUGTREE_ITEM_WORDS];
    if (it[0] == K_PROMPT_KV) p->splits_h[it[1]].nsplit = std::max(p->splits_h[it[1]].nsplit, it[4] + 1);
  }
  p->part_rows = 0;
  for (int g = 0; g < p->n_groups; ++g) {
    SplitInfo& s = p->splits_h[g];
    s.part_row0 = p->part_rows;
    if (s.nsplit > 1) p->part_rows += (int64_t)s.nsplit * p->groups_h[g].lp;
  }
  // Replay forward split-KV: per response query tile, its split count and chunk (the
  // cost of its split 0) from the queue, and the first of its Hq * nsplit partial slots.
  // (Tensor-core family only: its replay query tiles are the 128-row statistics tiles.)
  p->fsplit_h.assign(std::max(1, p->ntiles_r), FwdSplit{1, 0, 0});
  const size_t n_fwd_items = p->family == AUGTREE_KERNEL_TC ? p->n_items[AUGTREE_OP_REPLAY_FWD] : 0;
  for (size_t i = 0; i < n_fwd_items; ++i) {
    const int32_t* it = &p->queue_h[AUGTREE_OP_REPLAY_FWD][i * AUGTREE_ITEM_WORDS];
    FwdSplit& f = p->fsplit_h[p->groups_h[it[1]].tr0 + it[2]];
    f.nsplit = std::max(f.nsplit, it[4] + 1);
    if (it[4] == 0) f.chunk = it[5];
  }
  bool any_split = false;
  for (int g = 0; g < p->n_groups && n_fwd_items > 0; ++g)
    for (int32_t t = 0; t < (int32_t)cdiv(p->groups_h[g].lr, kFwdPartRows); ++t) {
      FwdSplit& f = p->fsplit_h[p->groups_h[g].tr0 + t];
      if (f.nsplit <= 1) continue;
      any_split = true;
      f.slot0 = p->n_fwd_parts;
      p->n_fwd_parts += (int64_t)cfg->hq * f.nsplit;
      p->fsplit_tiles_h.push_back(g);
      p->fsplit_tiles_h.push_back(t);
    }
  // Device copies.
  auto up = [&](void** dst, const void* src, size_t bytes) -> bool {
    if (bytes == 0) bytes = 16;
    if (cudaMalloc(dst, bytes) != cudaSuccess) return false;
    return cudaMemcpy(*dst, src, bytes, cudaMemcpyHostToDevice) == cudaSuccess;
  };
  bool ok = true;
  std::vector<int32_t> pad(4, 0);
  ok = ok && up((void**)&p->groups_d, p->groups_h.empty() ? (const void*)pad.data() : p->groups_h.data(),
                p->groups_h.size() * sizeof(GroupInfo));
  ok = ok && up((void**)&p->row_bstart_d, bstart.data(), bstart.size() * sizeof(int32_t));
  ok = ok && up((void**)&p->row_bend_d, bend.data(), bend.size() * sizeof(int32_t));
  // Error block: word 0 error bits, word 1 reserved, words 2-3 the wait limit (ns),
  // words 4-7 the persistent forward's work counters (zero).
  const uint64_t lim = kDefaultWaitLimitNs;
  uint32_t err_init[kErrBlockWords] = {};
  err_init[2] = (uint32_t)lim;
  err_init[3] = (uint32_t)(lim >> 32);
  ok = ok && up((void**)&p->err_d, err_init, sizeof(err_init));
  ok = ok && up((void**)&p->splits_d, p->splits_h.data(), p->splits_h.size() * sizeof(SplitInfo));
  if (any_split) {
    ok = ok && up((void**)&p->fsplit_d, p->fsplit_h.data(), p->fsplit_h.size() * sizeof(FwdSplit));
    ok = ok && up((void**)&p->fsplit_tiles_d, p->fsplit_tiles_h.data(), p->fsplit_tiles_h.size() * sizeof(int32_t));
  }
  for (int op = 0; op < kNumOps && ok; ++op)
    ok = up((void**)&p->queue_d[op], p->queue_h[op].empty() ? (const void*)pad.data() : p->queue_h[op].data(),
            p->queue_h[op].size() * sizeof(int32_t));
  auto up_lanes = [&](LaneSet& l) -> bool {
    if (l.off.empty()) return true;
    return up((void**)&l.off_d, l.off.data(), l.off.size() * sizeof(int32_t)) &&
           up((void**)&l.units_d, l.units.empty() ? (const void*)pad.data() : l.units.data(),
              l.units.size() * sizeof(int32_t));
  };
  for (int op = 0; op < 2 && ok; ++op) ok = up_lanes(p->lanes_dq[op]);
  for (int op = 0; op < kNumOps && ok; ++op) ok = up_lanes(p->lanes_kv[op]);
  if (!ok) {
    cudaGetLastError();
    augtree_plan_destroy(p);
    return AUGTREE_ERR_CUDA;
  }
  // The allocation-free prefill backward's scratch array: its device address on this
  // device, looked up here so that the call itself never loads a module or allocates.
  // A failed lookup only disables that entry point (it then returns AUGTREE_ERR_CUDA).
  if (static_scratch_address(&p->static_scratch) != cudaSuccess) {
    cudaGetLastError();
    p->static_scratch = nullptr;
  }
  *out = p;
  return AUGTREE_OK;
}

augtree_status augtree_plan_workspace_bytes(const augtree_plan* p, int32_t op, size_t* bytes) {
  if (!p || !bytes) return AUGTREE_ERR_INVALID_ARG;
  switch (op) {
    case AUGTREE_OP_PREFILL_FWD: *bytes = 0; return AUGTREE_OK;
    case AUGTREE_OP_REPLAY_FWD: *bytes = replay_fwd_ws(p).total; return AUGTREE_OK;
    case AUGTREE_OP_REPLAY_BWD: *bytes = replay_bwd_ws(p).total; return AUGTREE_OK;
    case AUGTREE_OP_PREFILL_BWD: *bytes = prefill_bwd_ws(p).total; return AUGTREE_OK;
    case AUGTREE_OP_TREE_BWD: *bytes = tree_bwd_ws(p).total; return AUGTREE_OK;
  }
  return AUGTREE_ERR_INVALID_ARG;
}

augtree_status augtree_schedule_export(const augtree_plan* p, int32_t op, int32_t* host_out, size_t cap_items,
                                       size_t* n_items) {
  if (!p || !n_items || op < 0 || op >= kNumOps) return AUGTREE_ERR_INVALID_ARG;
  *n_items = p->n_items[op];
  if (p->n_items[op] > cap_items) return AUGTREE_ERR_CAPACITY;
  if (p->n_items[op] == 0) return AUGTREE_OK;
  if (!host_out) return AUGTREE_ERR_INVALID_ARG;
  // Read back the device copy: the export shows what the kernels walk.
  if (cudaMemcpy(host_out, p->queue_d[op], p->n_items[op] * AUGTREE_ITEM_WORDS * sizeof(int32_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return AUGTREE_ERR_CUDA;
  return AUGTREE_OK;
}

}  // extern "C"

namespace {

augtree_status check_device(const augtree_plan* p) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return AUGTREE_ERR_CUDA;
  return cur == p->device ? AUGTREE_OK : AUGTREE_ERR_INVALID_ARG;
}

augtree_status from_cuda(cudaError_t e) { return e == cudaSuccess ? AUGTREE_OK : AUGTREE_ERR_CUDA; }

}  // namespace

extern "C" {

augtree_status augtree_prefill_fwd(const augtree_plan* p, const void* qp, const void* kp, const void* vp, void* op,
                                   float* lse_p, void* ws, size_t ws_bytes, void* stream) {
  (void)ws;
  (void)ws_bytes;
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_prompt > 0 && (!qp || !kp || !vp || !op || !lse_p)) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (p->n_items[AUGTREE_OP_PREFILL_FWD] == 0) return AUGTREE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  CallTimer tm(p, AUGTREE_OP_PREFILL_FWD, s);
  cudaError_t e;
  if (p->family == AUGTREE_KERNEL_TC) {
    tm.mark(AUGTREE_KID_FWD_TC);
    e = tc_fwd(p, AUGTREE_OP_PREFILL_FWD, qp, kp, vp, nullptr, nullptr, op, lse_p, nullptr, nullptr, s);
  } else {
    tm.mark(AUGTREE_KID_FWD_SIMT);
    e = simt_fwd(p, AUGTREE_OP_PREFILL_FWD, qp, kp, vp, nullptr, nullptr, op, lse_p, s);
  }
  tm.finish();
  return from_cuda(e);
}

augtree_status augtree_replay_fwd(const augtree_plan* p, const void* qr, const void* kp, const void* vp,
                                  const void* kr, const void* vr, void* or_, float* lse_r, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_resp > 0 && (!qr || !kr || !vr || !or_ || !lse_r)) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_resp > 0 && p->total_prompt > 0 && (!kp || !vp)) return AUGTREE_ERR_INVALID_ARG;
  const FwdWorkspace w = replay_fwd_ws(p);
  if (ws_bytes < w.total) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  if (w.total > 0 && (!ws || ((uintptr_t)ws & 15u))) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (p->n_items[AUGTREE_OP_REPLAY_FWD] == 0) return AUGTREE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  CallTimer tm(p, AUGTREE_OP_REPLAY_FWD, s);
  cudaError_t e;
  if (p->family == AUGTREE_KERNEL_TC) {
    // Split-KV (a queue too short for the GPU): the split tiles' partial states go to
    // the workspace and are merged in split order (Sec. 3.3).
    float* part_o = w.total ? (float*)((char*)ws + w.o_off) : nullptr;
    float* part_lse = w.total ? (float*)((char*)ws + w.lse_off) : nullptr;
    tm.mark(AUGTREE_KID_FWD_TC);
    e = tc_fwd(p, AUGTREE_OP_REPLAY_FWD, qr, kp, vp, kr, vr, or_, lse_r, part_o, part_lse, s);
    if (e == cudaSuccess && p->n_fwd_parts > 0) {
      tm.mark(AUGTREE_KID_FWD_MERGE);
      e = launch_fwd_split_merge(p, part_o, part_lse, or_, lse_r, s);
    }
  } else {
    tm.mark(AUGTREE_KID_FWD_SIMT);
    e = simt_fwd(p, AUGTREE_OP_REPLAY_FWD, qr, kp, vp, kr, vr, or_, lse_r, s);
  }
  tm.finish();
  return from_cuda(e);
}

augtree_status augtree_replay_bwd(const augtree_plan* p, const void* qr, const void* kp, const void* vp,
                                  const void* kr, const void* vr, const void* or_, const float* lse_r,
                                  const void* dor, void* dqr, void* dkr, void* dvr, float* dkp_sum,
                                  float* dvp_sum, void* ws, size_t ws_bytes, void* stream) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_resp > 0 && (!qr || !kr || !vr || !or_ || !lse_r || !dor || !dqr || !dkr || !dvr))
    return AUGTREE_ERR_INVALID_ARG;
  if (p->total_prompt > 0 && (!dkp_sum || !dvp_sum)) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_resp > 0 && p->total_prompt > 0 && (!kp || !vp)) return AUGTREE_ERR_INVALID_ARG;
  BwdWorkspace w = replay_bwd_ws(p);
  if (ws_bytes < w.total) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  if (w.total > 0 && (!ws || ((uintptr_t)ws & 15u))) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  float* delta = (float*)(base + w.delta_off);
  float* dq_acc = (float*)(base + w.dq_off);
  float* dk_part = (float*)(base + w.dkpart_off);
  float* dv_part = (float*)(base + w.dvpart_off);
  const int dt = p->cfg.dtype;
  cudaError_t e = cudaSuccess;
  const bool tc = p->family == AUGTREE_KERNEL_TC;
  CallTimer tm(p, AUGTREE_OP_REPLAY_BWD, s);
  if (tc) {
    // Key side (response dK/dV, prompt dK/dV summed over the branches), the split-K
    // reduction of the prompt partials, then the query side (dQ).
    void* aug = base + w.aug_off;
    if (p->total_resp > 0) {
      tm.mark(AUGTREE_KID_PREPROCESS);
      e = launch_preprocess_tiled(p, false, or_, dor, lse_r, delta, aug, s);
    }
    if (e == cudaSuccess && p->n_items[AUGTREE_OP_REPLAY_BWD] > 0) {
      tm.mark(AUGTREE_KID_BWD_KEY_SIDE);
      e = tc_bwd_kv(p, AUGTREE_OP_REPLAY_BWD, qr, dor, aug, nullptr, nullptr, nullptr, kp, vp, kr, vr, dkr, dvr,
                    nullptr, nullptr, dk_part, dv_part, dkp_sum, dvp_sum, nullptr, nullptr,
                    (float*)(base + w.slots_off), s);
    }
    if (e == cudaSuccess && p->total_prompt > 0) {
      tm.mark(AUGTREE_KID_SPLIT_REDUCE);
      e = launch_split_reduce(p, dk_part, dv_part, dkp_sum, dvp_sum, s);
    }
    if (e == cudaSuccess && p->total_resp > 0) {
      float* dq_part = (float*)(base + w.dqpart_off);
      tm.mark(AUGTREE_KID_BWD_QUERY_SIDE);
      e = tc_bwd_dq(p, AUGTREE_OP_REPLAY_BWD, qr, kp, vp, kr, vr, delta, dor, dqr, dq_part, s);
      if (e == cudaSuccess && p->n_fwd_parts > 0) {
        tm.mark(AUGTREE_KID_DQ_REDUCE);
        e = launch_dq_split_reduce(p, dq_part, dqr, s);
      }
    }
    tm.finish();
    return from_cuda(e);
  }
  if (p->total_resp > 0) {
    tm.mark(AUGTREE_KID_PREPROCESS);
    e = launch_preprocess(or_, dor, dt, p->total_resp, p->cfg.hq, p->cfg.head_dim, delta, dq_acc, s);
  }
  if (e == cudaSuccess && p->n_items[AUGTREE_OP_REPLAY_BWD] > 0) {
    tm.mark(AUGTREE_KID_BWD_SIMT);
    e = simt_bwd(p, AUGTREE_OP_REPLAY_BWD, qr, kp, vp, kr, vr, lse_r, dor, delta, dq_acc, dkr, dvr, dk_part,
                 dv_part, dkp_sum, dvp_sum, nullptr, nullptr, s);
  }
  if (e == cudaSuccess && p->total_prompt > 0) {
    tm.mark(AUGTREE_KID_SPLIT_REDUCE);
    e = launch_split_reduce(p, dk_part, dv_part, dkp_sum, dvp_sum, s);
  }
  if (e == cudaSuccess && p->total_resp > 0) {
    tm.mark(AUGTREE_KID_DQ_CONVERT);
    e = launch_dq_convert(dq_acc, dqr, dt, (int64_t)p->total_resp * p->cfg.hq * p->cfg.head_dim, s);
  }
  tm.finish();
  return from_cuda(e);
}

augtree_status augtree_prefill_bwd(const augtree_plan* p, const void* qp, const void* kp, const void* vp,
                                   const void* op, const float* lse_p, const void* dop, const float* dkp_acc,
                                   const float* dvp_acc, void* dqp, void* dkp, void* dvp, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_prompt > 0 && (!qp || !kp || !vp || !op || !lse_p || !dop || !dqp || !dkp || !dvp))
    return AUGTREE_ERR_INVALID_ARG;
  if ((dkp_acc == nullptr) != (dvp_acc == nullptr)) return AUGTREE_ERR_INVALID_ARG;
  BwdWorkspace w = prefill_bwd_ws(p);
  if (ws_bytes < w.total) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  if (w.total > 0 && (!ws || ((uintptr_t)ws & 15u))) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (p->total_prompt == 0) return AUGTREE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  float* delta = (float*)(base + w.delta_off);
  float* dq_acc = (float*)(base + w.dq_off);
  const int dt = p->cfg.dtype;
  const bool tc = p->family == AUGTREE_KERNEL_TC;
  CallTimer tm(p, AUGTREE_OP_PREFILL_BWD, s);
  if (tc) {
    void* aug = base + w.aug_off;
    tm.mark(AUGTREE_KID_PREPROCESS);
    cudaError_t e = launch_preprocess_tiled(p, true, op, dop, lse_p, delta, aug, s);
    if (e == cudaSuccess) {
      tm.mark(AUGTREE_KID_BWD_KEY_SIDE);
      e = tc_bwd_kv(p, AUGTREE_OP_PREFILL_BWD, qp, dop, aug, nullptr, nullptr, nullptr, kp, vp, nullptr, nullptr, dkp,
                    dvp, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dkp_acc, dvp_acc,
                    (float*)(base + w.slots_off), s);
    }
    if (e == cudaSuccess) {
      tm.mark(AUGTREE_KID_BWD_QUERY_SIDE);
      e = tc_bwd_dq(p, AUGTREE_OP_PREFILL_BWD, qp, kp, vp, nullptr, nullptr, delta, dop, dqp, nullptr, s);
    }
    tm.finish();
    return from_cuda(e);
  }
  tm.mark(AUGTREE_KID_PREPROCESS);
  cudaError_t e = launch_preprocess(op, dop, dt, p->total_prompt, p->cfg.hq, p->cfg.head_dim, delta, dq_acc, s);
  if (e == cudaSuccess && p->n_items[AUGTREE_OP_PREFILL_BWD] > 0) {
    tm.mark(AUGTREE_KID_BWD_SIMT);
    e = simt_bwd(p, AUGTREE_OP_PREFILL_BWD, qp, kp, vp, nullptr, nullptr, lse_p, dop, delta, dq_acc, dkp, dvp,
                 nullptr, nullptr, nullptr, nullptr, dkp_acc, dvp_acc, s);
  }
  if (e == cudaSuccess) {
    tm.mark(AUGTREE_KID_DQ_CONVERT);
    e = launch_dq_convert(dq_acc, dqp, dt, (int64_t)p->total_prompt * p->cfg.hq * p->cfg.head_dim, s);
  }
  tm.finish();
  return from_cuda(e);
}

augtree_status augtree_tree_bwd(const augtree_plan* p, const void* qp, const void* kp, const void* vp, const void* op,
                                const float* lse_p, const void* dop, const void* qr, const void* kr, const void* vr,
                                const void* or_, const float* lse_r, const void* dor, void* dqp, void* dkp, void* dvp,
                                void* dqr, void* dkr, void* dvr, void* ws, size_t ws_bytes, void* stream) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  if (p->total_prompt > 0 && (!qp || !kp || !vp || !op || !lse_p || !dop || !dqp || !dkp || !dvp))
    return AUGTREE_ERR_INVALID_ARG;
  if (p->total_resp > 0 && (!qr || !kr || !vr || !or_ || !lse_r || !dor || !dqr || !dkr || !dvr))
    return AUGTREE_ERR_INVALID_ARG;
  const TreeWorkspace w = tree_bwd_ws(p);
  if (ws_bytes < w.total) return AUGTREE_ERR_WORKSPACE_TOO_SMALL;
  if (w.total > 0 && (!ws || ((uintptr_t)ws & 15u))) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  char* base = (char*)ws;
  if (p->family != AUGTREE_KERNEL_TC) {
    // SIMT family: the two calls, with the replay sums in the workspace.
    float* dks = (float*)(base + w.sum_off);
    float* dvs = (float*)(base + w.sum_off + w.sum_bytes);
    st = augtree_replay_bwd(p, qr, kp, vp, kr, vr, or_, lse_r, dor, dqr, dkr, dvr, p->total_prompt ? dks : nullptr,
                            p->total_prompt ? dvs : nullptr, base, w.r.total, stream);
    if (st != AUGTREE_OK) return st;
    return augtree_prefill_bwd(p, qp, kp, vp, op, lse_p, dop, p->total_prompt ? dks : nullptr,
                               p->total_prompt ? dvs : nullptr, dqp, dkp, dvp, base + w.p_off, w.p.slots_off, stream);
  }
  cudaStream_t s = (cudaStream_t)stream;
  float* delta_r = (float*)(base + w.r.delta_off);
  void* aug_r = base + w.r.aug_off;
  float* delta_p = (float*)(base + w.p_off + w.p.delta_off);
  void* aug_p = base + w.p_off + w.p.aug_off;
  float* dk_part = (float*)(base + w.r.dkpart_off);
  float* dv_part = (float*)(base + w.r.dvpart_off);
  cudaError_t e = cudaSuccess;
  CallTimer tm(p, AUGTREE_OP_TREE_BWD, s);
  // Row statistics of both sides, then one key-side pass: every prompt KV tile walks its
  // prompt's own causal query tiles and all branches' query tiles in one accumulator
  // (split-K partials only where the prompt has few tiles), every response KV tile its
  // branch's tiles; then the query side of both.
  if (p->total_resp > 0) {
    tm.mark(AUGTREE_KID_PREPROCESS);
    e = launch_preprocess_tiled(p, false, or_, dor, lse_r, delta_r, aug_r, s);
  }
  if (e == cudaSuccess && p->total_prompt > 0) {
    tm.mark(AUGTREE_KID_PREPROCESS);
    e = launch_preprocess_tiled(p, true, op, dop, lse_p, delta_p, aug_p, s);
  }
  if (e == cudaSuccess && p->n_items[AUGTREE_OP_TREE_BWD] > 0) {
    tm.mark(AUGTREE_KID_BWD_KEY_SIDE);
    e = tc_bwd_kv(p, AUGTREE_OP_TREE_BWD, qr, dor, aug_r, qp, dop, aug_p, kp, vp, kr, vr, dkr, dvr, dkp, dvp,
                  dk_part, dv_part, nullptr, nullptr, nullptr, nullptr, (float*)(base + w.r.slots_off), s);
  }
  if (e == cudaSuccess && p->part_rows > 0) {
    tm.mark(AUGTREE_KID_SPLIT_REDUCE);
    e = launch_split_reduce_final(p, dk_part, dv_part, dkp, dvp, s);
  }
  if (e == cudaSuccess && p->total_prompt > 0) {
    tm.mark(AUGTREE_KID_BWD_QUERY_SIDE);
    e = tc_bwd_dq(p, AUGTREE_OP_PREFILL_BWD, qp, kp, vp, nullptr, nullptr, delta_p, dop, dqp, nullptr, s);
  }
  if (e == cudaSuccess && p->total_resp > 0) {
    float* dq_part = (float*)(base + w.r.dqpart_off);
    tm.mark(AUGTREE_KID_BWD_QUERY_SIDE);
    e = tc_bwd_dq(p, AUGTREE_OP_REPLAY_BWD, qr, kp, vp, kr, vr, delta_r, dor, dqr, dq_part, s);
    if (e == cudaSuccess && p->n_fwd_parts > 0) {
      tm.mark(AUGTREE_KID_DQ_REDUCE);
      e = launch_dq_split_reduce(p, dq_part, dqr, s);
    }
  }
  tm.finish();
  return from_cuda(e);
}

augtree_status augtree_plan_set_timing(augtree_plan* p, int32_t enable) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (enable && !p->timing.created) {
    for (int op = 0; op < kNumOps; ++op)
      for (int c = 0; c < AUGTREE_TIMING_RING; ++c)
        for (int k = 0; k < augtree_plan::kTimingMarks; ++k)
          if (cudaEventCreate(&p->timing.ev[op][c][k]) != cudaSuccess) return AUGTREE_ERR_CUDA;
    p->timing.created = true;
  }
  p->timing.on = enable != 0;
  return AUGTREE_OK;
}

augtree_status augtree_plan_kernel_times(const augtree_plan* p, int32_t op, int32_t back, int32_t* kind, float* ms,
                                         int32_t cap, int32_t* n) {
  if (!p || !n || op < 0 || op >= kNumOps || back < 0 || back >= AUGTREE_TIMING_RING || cap < 0) return AUGTREE_ERR_INVALID_ARG;
  const auto& T = p->timing;
  if (!T.on || T.calls[op] <= (uint32_t)back) return AUGTREE_ERR_INVALID_ARG;
  if (cap > 0 && (!kind || !ms)) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  const int slot = (int)((T.calls[op] - 1 - (uint32_t)back) % AUGTREE_TIMING_RING);
  const int kernels = T.n_marks[op][slot] - 1;
  if (cudaEventSynchronize(T.ev[op][slot][kernels]) != cudaSuccess) return AUGTREE_ERR_CUDA;
  int written = 0;
  for (int k = 0; k < kernels && written < cap; ++k) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, T.ev[op][slot][k], T.ev[op][slot][k + 1]) != cudaSuccess) return AUGTREE_ERR_CUDA;
    kind[written] = T.kind[op][slot][k];
    ms[written] = t;
    ++written;
  }
  *n = written;
  return AUGTREE_OK;
}

augtree_status augtree_plan_set_wait_limit(augtree_plan* p, uint64_t ns) {
  if (!p || ns == 0 || ns > kMaxWaitLimitNs) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (cudaMemcpy(p->err_d + 2, &ns, sizeof(ns), cudaMemcpyHostToDevice) != cudaSuccess) return AUGTREE_ERR_CUDA;
  return AUGTREE_OK;
}

augtree_status augtree_plan_check(const augtree_plan* p, void* stream) {
  if (!p) return AUGTREE_ERR_INVALID_ARG;
  augtree_status st = check_device(p);
  if (st != AUGTREE_OK) return st;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return AUGTREE_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpy(&w, p->err_d, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return AUGTREE_ERR_CUDA;
  if (w != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(p->err_d, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return AUGTREE_ERR_CUDA;
    return (w & 1u) ? AUGTREE_ERR_TIMEOUT : AUGTREE_ERR_DEVICE_CHECK;
  }
  return AUGTREE_OK;
}

augtree_status augtree_lse_merge(int64_t rows, int32_t h, int32_t d, const float* oa, const float* lse_a,
                                 const float* ob, const float* lse_b, float* o, float* lse, void* stream) {
  if (rows < 0 || h <= 0 || d <= 0) return AUGTREE_ERR_INVALID_ARG;
  if (rows == 0) return AUGTREE_OK;
  if (!oa || !lse_a || !ob || !lse_b || !o || !lse) return AUGTREE_ERR_INVALID_ARG;
  return from_cuda(launch_lse_merge(rows, h, d, oa, lse_a, ob, lse_b, o, lse, (cudaStream_t)stream));
}

augtree_status augtree_lse_merge_bwd(int64_t rows, int32_t h, int32_t d, const float* oa, const float* lse_a,
                                     const float* ob, const float* lse_b, const float* dout, const float* dlse,
                                     float* doa, float* dlse_a, float* dob, float* dlse_b, void* stream) {
  if (rows < 0 || h <= 0 || d <= 0) return AUGTREE_ERR_INVALID_ARG;
  if (rows == 0) return AUGTREE_OK;
  if (!oa || !lse_a || !ob || !lse_b || !dout || !doa || !dlse_a || !dob || !dlse_b) return AUGTREE_ERR_INVALID_ARG;
  return from_cuda(launch_lse_merge_bwd(rows, h, d, oa, lse_a, ob, lse_b, dout, dlse, doa, dlse_a, dob, dlse_b,
                                        (cudaStream_t)stream));
}

}  // extern "C"
