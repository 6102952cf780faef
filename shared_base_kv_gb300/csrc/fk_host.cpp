// Host side of libforkkv: pool metadata (page reference counts and free
// list, copy-on-write appends, agent registry, rCache arena), the work-list
// planner, and the C ABI.  Kernels live in fk_kernels.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "fk_internal.h"

using namespace fk;

namespace {

thread_local std::string g_err;

fk_status fail(fk_status code, const std::string& msg) {
  g_err = msg;
  return code;
}

fk_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FK_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct HostPlan {
  std::vector<fk_work_item> items;
  std::vector<int32_t> row_agent, row_cg, pages, tile_agents;
  std::vector<int32_t> csr_ptr, csr_slots;
  std::vector<int32_t> cta_begin;   // items [cta_begin[c], cta_begin[c+1]) run on CTA c
  int n_partials = 0;
  std::vector<MPair> mpairs;        // four-agent decode calls: one M per (agent tile, kv head)
  std::vector<int32_t> item_mpair;  // per item: its M pair
};

// Pinned host staging buffer for small host->device uploads.  A new upload
// waits for the previous one to have been consumed.
struct Staging {
  void* host = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
  bool pending = false;
};

}  // namespace

struct fk_pool {
  fk_pool_config cfg;
  PoolGeom g;
  uint64_t uid = 0;                          // unique per pool of the process (never reused)
  int device = 0;
  int num_sms = 0;
  // decode-shaped calls with d = 128 on the uncompressed pool: tiles of
  // eight agent slots (FORKKV_DECODE_SLOTS=8 at pool creation) instead of
  // four agents
  bool slots8 = false;
  bool stall_probe = false;                  // failure-detection test hook (fk_pool_set_test_stall)
  std::vector<int32_t> refcount;             // per page
  std::vector<int32_t> free_list;            // stack of free page ids
  std::vector<uint8_t> fill;                 // [L][num_pages] tokens held
  struct Agent {
    bool live = false;
    int rank = 0, rp = 0;
    float s = 0.f;
    int64_t rc_off = 0, rc_bytes = 0;
  };
  std::vector<Agent> agents;
  std::map<int64_t, int64_t> rc_free;        // offset -> bytes
  std::map<int64_t, int> rc_users;           // rCache offset -> agents reading it (Shared-A)
  Staging stage;
  // cached work list
  bool plan_valid = false;
  uint64_t plan_gen = 0;                     // bumped whenever agents or pages change
  std::vector<int32_t> key;                  // call inputs the plan is for
  HostPlan plan;
  PlanDev plan_dev{};
  int last_launches = 0;
  void* profile_event = nullptr;
};

namespace {

fk_status validate_config(const fk_pool_config* c) {
  if (!c) return fail(FK_ERR_INVALID_ARG, "config is NULL");
  if (c->n_layers < 1) return fail(FK_ERR_INVALID_ARG, "n_layers must be >= 1");
  if (c->n_kv_heads < 1 || c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads)
    return fail(FK_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(FK_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->page_size != kPage) return fail(FK_ERR_UNSUPPORTED, "page_size must be 16");
  if (c->num_pages < 1) return fail(FK_ERR_INVALID_ARG, "num_pages must be >= 1");
  if (c->max_agents < 1) return fail(FK_ERR_INVALID_ARG, "max_agents must be >= 1");
  if (c->max_rank < 8 || c->max_rank > kMaxRankPad || c->max_rank % 8)
    return fail(FK_ERR_UNSUPPORTED, "max_rank must be a multiple of 8 in [8, 64]");
  if (c->max_tokens < 1) return fail(FK_ERR_INVALID_ARG, "max_tokens must be >= 1");
  if (c->rcache_rank_budget < 0 || c->workspace_bytes < 0)
    return fail(FK_ERR_INVALID_ARG, "negative arena size");
  if (!(c->rope_base > 1.0f)) return fail(FK_ERR_INVALID_ARG, "rope_base must be > 1");
  return FK_OK;
}

PoolGeom make_geom(const fk_pool_config* c) {
  PoolGeom g{};
  g.L = c->n_layers;
  g.H_q = c->n_q_heads;
  g.H_kv = c->n_kv_heads;
  g.d = c->head_dim;
  g.G = c->n_q_heads / c->n_kv_heads;
  g.num_pages = c->num_pages;
  g.max_agents = c->max_agents;
  g.rmax_pad = rank_pad(c->max_rank);
  g.tcap = (int32_t)align_up(c->max_tokens, kTileTok);
  g.rope_base = c->rope_base;
  g.compressed = c->compressed ? 1 : 0;
  g.page_bytes = (int64_t)kPage * g.d * 2;
  g.kb_layer_bytes = (int64_t)g.num_pages * g.H_kv * g.page_bytes;
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    int64_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  g.off_kb = take(g.kb_layer_bytes * g.L);
  g.off_vb = take(g.kb_layer_bytes * g.L);
  int64_t budget = c->rcache_rank_budget ? c->rcache_rank_budget
                                         : (int64_t)c->max_agents * c->max_rank;
  // rank budget in padded-rank units: every agent may round up to 16
  int64_t budget_pad = align_up(budget, 16) + 16LL * c->max_agents;
  budget_pad = std::min<int64_t>(budget_pad, (int64_t)c->max_agents * g.rmax_pad);
  int64_t rc_bytes = budget_pad * g.L * 2LL * g.tcap * 2;
  int64_t off_rc = take(rc_bytes);
  (void)off_rc;  // arena starts here; recorded below via off_bk - rc_bytes
  g.bk_agent_bytes = (int64_t)g.L * g.H_kv * g.d * g.rmax_pad * 2;
  g.bv_agent_bytes = (int64_t)g.L * g.rmax_pad * g.H_kv * g.d * 2;
  g.off_bk = take(g.bk_agent_bytes * g.max_agents);
  g.off_bv = take(g.bv_agent_bytes * g.max_agents);
  g.off_agents = take((int64_t)sizeof(AgentDev) * g.max_agents);
  g.off_rope = take(4LL * 4 * 64);
  g.off_err = take(64);
  g.off_lvmap = take(128LL * g.max_agents);
  // the eight-slot decode kernel reads each key's RoPE rotations from here
  g.off_trig = g.d == 128 ? take((int64_t)g.tcap * (g.d / 2) * 4) : -1;
  if (g.compressed) {
    int64_t tok = (int64_t)g.L * g.num_pages * g.H_kv * kPage;
    g.off_kq = take(tok * g.d);
    g.off_vc = take(tok * (3 * g.d / 8));
    g.off_vn = take(tok * 4);
    g.off_ks = take(4LL * g.L);
    g.off_kmax = take(4LL * g.L);
  } else {
    g.off_kq = g.off_vc = g.off_vn = g.off_ks = g.off_kmax = -1;
  }
  g.meta_bytes = align_up(8LL * g.num_pages + 4096, 256);
  g.off_meta = take(g.meta_bytes);
  g.ws_bytes = c->workspace_bytes ? c->workspace_bytes : (64LL << 20);
  g.off_ws = take(g.ws_bytes);
  return g;
}

int64_t total_bytes(const PoolGeom& g) { return g.off_ws + g.ws_bytes; }

int64_t rc_arena_offset(const PoolGeom& g) {
  // the rCache arena sits right after the value pages
  return align_up(g.off_vb + g.kb_layer_bytes * g.L, 256);
}
int64_t rc_arena_bytes(const PoolGeom& g) { return g.off_bk - rc_arena_offset(g); }

fk_status stage_upload(fk_pool* p, const void* src, size_t bytes, void* dst,
                       cudaStream_t st) {
  Staging& s = p->stage;
  if (s.pending) {
    cudaError_t e = cudaEventSynchronize(s.done);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    s.pending = false;
  }
  if (bytes > s.cap) {
    if (s.host) cudaFreeHost(s.host);
    s.host = nullptr;
    size_t cap = std::max<size_t>(bytes, 1 << 20);
    cudaError_t e = cudaMallocHost(&s.host, cap);
    if (e != cudaSuccess) { s.cap = 0; return cuda_fail(e, "cudaMallocHost"); }
    s.cap = cap;
  }
  std::memcpy(s.host, src, bytes);
  cudaError_t e = cudaMemcpyAsync(dst, s.host, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  e = cudaEventRecord(s.done, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  s.pending = true;
  return FK_OK;
}

// TMA tensor map of one agent's Lv rows, all layers.  Lv of layer l sits at
// rc_off + l * rc_layer_bytes + tcap * rp * 2 as [tcap/8 chunks][rp/8 rank
// groups][8 ranks][8 keys] (bf16); the map's dimensions, innermost first,
// are (key in chunk, rank in group, rank group, chunk, layer), so a box of
// (8, 8, 1, 16, 1) is one rank group of a 128-key tile: 16 consecutive
// 128-byte core matrices (keys past tcap read as zeros).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  });
  return fn;
}

static fk_status encode_lv_map(const PoolGeom& g, const fk_pool::Agent& A, CUtensorMap* m) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return fail(FK_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  void* base = g.base + A.rc_off + (int64_t)g.tcap * A.rp * 2;
  const cuuint64_t dims[5] = {8, 8, (cuuint64_t)(A.rp / 8), (cuuint64_t)(g.tcap / 8),
                              (cuuint64_t)g.L};
  const cuuint64_t strides[4] = {16, 128, (cuuint64_t)A.rp * 16,
                                 (cuuint64_t)rc_layer_bytes(g, A.rp)};
  const cuuint32_t box[5] = {8, 8, 1, 16, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FK_ERR_CUDA, "cuTensorMapEncodeTiled failed for an Lv map");
  return FK_OK;
}

fk_status upload_agent(fk_pool* p, int a, cudaStream_t st) {
  const auto& A = p->agents[a];
  AgentDev dv{};
  dv.rp = A.live ? A.rp : 0;
  dv.s = A.s;
  dv.rc_off = A.rc_off;
  fk_status r = stage_upload(p, &dv, sizeof(dv),
                             p->g.base + p->g.off_agents + (int64_t)a * sizeof(AgentDev), st);
  if (r != FK_OK || !A.live) return r;
  alignas(64) CUtensorMap m;
  r = encode_lv_map(p->g, A, &m);
  if (r != FK_OK) return r;
  return stage_upload(p, &m, sizeof(m), p->g.base + p->g.off_lvmap + 128LL * a, st);
}

// ----------------------------------------------------------- planner --

// slots8: the eight-slot tiles of the decode kernel for decode-shaped calls
// (fk_decode8.cu): two halves of at most four agents and 64 padded ranks
// each, agent slot s holding tile rows 4 s .. 4 s + 3; empty slots are -1
// in tile_agents and their rows -1 in row_agent (no output row reads them).
fk_status plan_build(int A, int C, int H_q, int H_kv, int P, const int32_t* bt,
                     int max_pages, const int32_t* seq, const int32_t* rpad,
                     int max_rows, int max_rank_sum, int target_items,
                     HostPlan& out, bool slots8 = false) {
  if (A < 1 || C < 1) return fail(FK_ERR_INVALID_ARG, "A and C must be >= 1");
  if (H_kv < 1 || H_q % H_kv) return fail(FK_ERR_INVALID_ARG, "bad head counts");
  if (!bt || !seq || !rpad) return fail(FK_ERR_INVALID_ARG, "NULL table");
  if (max_rows < 1 || max_rows > kMaxRows || max_rank_sum < 16)
    return fail(FK_ERR_INVALID_ARG, "bad tile limits");
  const int G = H_q / H_kv;
  for (int i = 0; i < A; ++i) {
    if (seq[i] < C) return fail(FK_ERR_INVALID_ARG, "seq_lens[i] must be >= C >= 1");
    int np = (seq[i] + P - 1) / P;
    if (np > max_pages) return fail(FK_ERR_INVALID_ARG, "seq_len exceeds max_pages");
    for (int lp = 0; lp < np; ++lp)
      if (bt[(int64_t)i * max_pages + lp] < 0)
        return fail(FK_ERR_INVALID_ARG, "block table names no page for a live token");
    if (rpad[i] < 16 || rpad[i] % 16 || rpad[i] > kMaxRankPad)
      return fail(FK_ERR_INVALID_ARG, "bad padded rank");
  }
  // 1. sharing classes: (logical page, physical page) -> agents
  std::map<std::pair<int32_t, int32_t>, std::vector<int32_t>> cls;
  for (int i = 0; i < A; ++i) {
    int np = (seq[i] + P - 1) / P;
    for (int lp = 0; lp < np; ++lp)
      cls[{lp, bt[(int64_t)i * max_pages + lp]}].push_back(i);
  }
  // 2. group by agent set; pages of a set in logical order
  std::map<std::vector<int32_t>, std::vector<std::pair<int32_t, int32_t>>> sets;
  for (auto& kv : cls) sets[kv.second].push_back(kv.first);
  // 3. tiles of every set, and page runs
  if (slots8 && G * C != 4) return fail(FK_ERR_INVALID_ARG, "eight-slot tiles need four rows per agent");
  struct Tile { std::vector<int32_t> agents; std::vector<std::pair<int32_t,int32_t>> rows; int rank_sum; int n_real = 0; };
  struct SetWork { std::vector<Tile> tiles; std::vector<std::vector<std::pair<int32_t,int32_t>>> runs; };
  std::vector<SetWork> work;
  int64_t total_units = 0;
  const int rpa = G * C;
  for (auto& kv : sets) {
    SetWork sw;
    Tile cur{{}, {}, 0};
    auto flush = [&]() { if (!cur.rows.empty()) sw.tiles.push_back(cur); cur = Tile{{}, {}, 0}; };
    // 16-row groups touched by the agents of a tile, each agent counted once
    auto groups_with = [&](int n_agents) {
      int tot = 0;
      for (int k = 0; k < n_agents; ++k) tot += (k * rpa + rpa - 1) / 16 - (k * rpa) / 16 + 1;
      return tot;
    };
    if (slots8) {
      // fill half 0, then half 1; an agent that does not fit the current
      // half opens the next one (or a new tile)
      int half = 0, nh[2] = {0, 0}, rh[2] = {0, 0};
      std::vector<int32_t> slot(kDecodeSlots, -1);
      auto emit = [&]() {
        if (nh[0] + nh[1] == 0) return;
        Tile t{{}, {}, rh[0] + rh[1], nh[0] + nh[1]};
        for (int s2 = 0; s2 < kDecodeSlots; ++s2) {
          t.agents.push_back(slot[s2]);
          for (int g2 = 0; g2 < rpa; ++g2) t.rows.push_back({slot[s2], slot[s2] >= 0 ? g2 : 0});
        }
        sw.tiles.push_back(t);
        half = 0; nh[0] = nh[1] = 0; rh[0] = rh[1] = 0;
        std::fill(slot.begin(), slot.end(), -1);
      };
      for (int32_t a : kv.first) {
        while (true) {
          if (nh[half] < kDecodeSlots / 2 && rh[half] + rpad[a] <= kDecodeHalfRank) {
            slot[(kDecodeSlots / 2) * half + nh[half]] = a;
            ++nh[half];
            rh[half] += rpad[a];
            break;
          }
          if (half == 0) { half = 1; continue; }
          emit();
        }
      }
      emit();
    }
    // Four-agent decode tiles (four rows per agent): a tile's 128-key step
    // costs about the same whatever its agents, so the set's agents are
    // packed into as few tiles as the rank budget allows (largest rank
    // first, each into the first tile with room), and each tile's agents
    // are then ordered so that its two halves (agents 0-1 and 2-3, one
    // compute warpgroup each) carry ranks as even as possible.  Agents of
    // equal rank keep their call order.
    const bool pack = rpa == 4 && !slots8;
    std::vector<int32_t> order(kv.first.begin(), kv.first.end());
    if (pack)
      std::stable_sort(order.begin(), order.end(),
                       [&](int32_t x, int32_t y) { return rpad[x] > rpad[y]; });
    auto fits = [&](const Tile& t, int32_t a) {
      return ((int)t.agents.size() + 1) * rpa <= max_rows && t.rank_sum + rpad[a] <= max_rank_sum &&
             (int)t.agents.size() < kMaxAgentsPerTile &&
             groups_with((int)t.agents.size() + 1) <= kMaxRowGroups;
    };
    std::vector<Tile> packed;
    for (int32_t a : (slots8 ? std::vector<int32_t>{} : order)) {
      if (pack) {
        size_t ti = 0;
        while (ti < packed.size() && !fits(packed[ti], a)) ++ti;
        if (ti == packed.size()) packed.push_back(Tile{{}, {}, 0});
        Tile& t = packed[ti];
        t.agents.push_back(a);
        t.rank_sum += rpad[a];
        ++t.n_real;
      } else if (rpa <= max_rows) {
        if (!fits(cur, a)) flush();
        cur.agents.push_back(a);
        cur.rank_sum += rpad[a];
        ++cur.n_real;
        for (int cg = 0; cg < rpa; ++cg) cur.rows.push_back({a, cg});
      } else {
        flush();
        for (int c0 = 0; c0 < rpa; c0 += max_rows) {
          Tile t{{a}, {}, rpad[a], 1};
          for (int cg = c0; cg < std::min(rpa, c0 + max_rows); ++cg) t.rows.push_back({a, cg});
          sw.tiles.push_back(t);
        }
      }
    }
    if (!slots8) flush();
    for (Tile& t : packed) {
      // the slot order with the most even halves (the first such order in
      // lexicographic order of positions, so equal ranks keep call order)
      std::vector<int> perm(t.agents.size()), best;
      for (size_t k = 0; k < perm.size(); ++k) perm[k] = (int)k;
      int best_max = 1 << 30;
      do {
        int h[2] = {0, 0};
        for (size_t k = 0; k < perm.size(); ++k) h[k < 2 ? 0 : 1] += rpad[t.agents[perm[k]]];
        if (std::max(h[0], h[1]) < best_max) { best_max = std::max(h[0], h[1]); best = perm; }
      } while (std::next_permutation(perm.begin(), perm.end()));
      std::vector<int32_t> ag(t.agents.size());
      for (size_t k = 0; k < perm.size(); ++k) ag[k] = t.agents[best[k]];
      t.agents = ag;
      t.rows.clear();
      for (int32_t a : t.agents)
        for (int cg = 0; cg < rpa; ++cg) t.rows.push_back({a, cg});
      sw.tiles.push_back(t);
    }
    const auto& pg = kv.second;   // sorted by logical page
    size_t s0 = 0;
    for (size_t k = 1; k <= pg.size(); ++k) {
      if (k == pg.size() || pg[k].first != pg[k - 1].first + 1) {
        sw.runs.emplace_back(pg.begin() + s0, pg.begin() + k);
        total_units += (int64_t)(k - s0) * sw.tiles.size() * H_kv;
        s0 = k;
      }
    }
    work.push_back(std::move(sw));
  }
  // 4. emit items.  Segments = (tile, head, page run) in set / tile / head /
  // run order; their pages, weighted by the per-page work, are cut into
  // `target_items` contiguous pieces of equal weight, one per CTA.  A piece
  // that crosses segment boundaries becomes several items run back to back
  // by the same CTA.
  //
  // Per-page weight: the four-agent decode kernel's 128-key tile costs
  // about the same whatever its agents (its per-tile chain, not the
  // per-agent work, sets the pace; measured on GB300): about 1.9 us with at
  // most 32 padded ranks (one 128-column Z chunk) and 2.25 us with more:
  // weights 5 and 6.  (Tiles of one or two agents with 48 or more ranks
  // share their rank groups between both compute warpgroups; see the
  // decode kernel.)  For the other kernels the work
  // grows with the agents (base + one unit per agent).  A segment's last,
  // partial tile costs as much as a full one and is weighed as one.
  auto tile_wpp = [&](const Tile& t) -> int {
    if (rpa == 4 && !slots8) {
      int h0 = 0, h1 = 0;
      for (size_t k = 0; k < t.agents.size(); ++k) (k < 2 ? h0 : h1) += rpad[t.agents[k]];
      return h0 + h1 <= 32 ? 5 : 6;
    }
    return 2 + t.n_real;
  };
  auto full_tiles = [](int64_t pages) { return (pages + kTilePages - 1) / kTilePages * kTilePages; };
  (void)total_units;
  HostPlan pl;
  struct Seg { int tile_row0, tile_ag0, n_rows, n_ag, rank_sum, head, page0, lp0, len, wpp; };
  std::vector<Seg> segs;
  int64_t total_w = 0;
  for (auto& sw : work) {
    std::vector<int> tile_row0, tile_ag0;
    for (auto& t : sw.tiles) {
      tile_row0.push_back((int)pl.row_agent.size());
      for (auto& r : t.rows) { pl.row_agent.push_back(r.first); pl.row_cg.push_back(r.second); }
      tile_ag0.push_back((int)pl.tile_agents.size());
      for (int32_t a : t.agents) pl.tile_agents.push_back(a);
    }
    std::vector<int> run_page0;
    for (auto& run : sw.runs) {
      run_page0.push_back((int)pl.pages.size());
      for (auto& pr : run) pl.pages.push_back(pr.second);
    }
    for (size_t ti = 0; ti < sw.tiles.size(); ++ti)
      for (int h = 0; h < H_kv; ++h)
        for (size_t ri = 0; ri < sw.runs.size(); ++ri) {
          Seg sg{tile_row0[ti], tile_ag0[ti], (int)sw.tiles[ti].rows.size(),
                 (int)sw.tiles[ti].agents.size(), sw.tiles[ti].rank_sum, h, run_page0[ri],
                 sw.runs[ri][0].first, (int)sw.runs[ri].size(), tile_wpp(sw.tiles[ti])};
          segs.push_back(sg);
          total_w += full_tiles(sg.len) * sg.wpp;
        }
  }
  int64_t total_tiles = 0;
  for (auto& sg : segs) total_tiles += (sg.len + kTilePages - 1) / kTilePages;
  const int n_ctas = (int)std::max<int64_t>(1, std::min<int64_t>(target_items, total_tiles));
  auto push_item = [&](const Seg& sg, int off, int take) {
    fk_work_item it{};
    it.head = sg.head;
    it.row_begin = sg.tile_row0;
    it.n_rows = sg.n_rows;
    it.page_begin = sg.page0 + off;
    it.n_pages = take;
    it.lp_begin = sg.lp0 + off;
    it.agent_begin = sg.tile_ag0;
    it.n_agents = sg.n_ag;
    it.partial_begin = pl.n_partials;
    it.sum_rank = sg.rank_sum;
    pl.n_partials += it.n_rows;
    pl.items.push_back(it);
  };
  if (slots8 && (int64_t)segs.size() <= n_ctas) {
    // One item per CTA: every segment gets a share of the CTAs in
    // proportion to its tiles (at least one, at most one per tile), the
    // largest remainders first, and is cut into that many runs of whole
    // tiles of nearly equal length.  Each CTA then builds one M.
    const int ns = (int)segs.size();
    std::vector<int64_t> tiles(ns);
    std::vector<int> share(ns, 1);
    for (int i = 0; i < ns; ++i) tiles[i] = (segs[i].len + kTilePages - 1) / kTilePages;
    int used = ns;
    while (used < n_ctas) {
      int best = -1;
      double best_load = 0.0;
      for (int i = 0; i < ns; ++i) {
        if (share[i] >= tiles[i]) continue;
        const double load = (double)tiles[i] / share[i];
        if (best < 0 || load > best_load) { best = i; best_load = load; }
      }
      if (best < 0) break;
      ++share[best];
      ++used;
    }
    pl.cta_begin.clear();
    for (int i = 0; i < ns; ++i) {
      const Seg& sg = segs[i];
      for (int c = 0; c < share[i]; ++c) {
        const int64_t t0 = tiles[i] * c / share[i], t1 = tiles[i] * (c + 1) / share[i];
        const int off = (int)(t0 * kTilePages);
        const int take = (int)std::min<int64_t>(t1 * kTilePages, sg.len) - off;
        pl.cta_begin.push_back((int)pl.items.size());
        push_item(sg, off, take);
      }
    }
    pl.cta_begin.push_back((int)pl.items.size());
  } else {
    pl.cta_begin.assign(n_ctas + 1, 0);
    // A CTA that starts a second item pays for it (the item's set-up, its
    // own M and a drained pipeline: about two tiles of work), so such CTAs
    // are charged that much extra weight; pieces are cut at whole key tiles
    // of their segment, so only a segment's last item has a partial tile.
    auto item_cost = [&](const Seg& sg) { return (int64_t)2 * kTilePages * sg.wpp; };
    int64_t total_wc = total_w;
    for (size_t i = 1; i < segs.size(); ++i) total_wc += item_cost(segs[i]);
    size_t si = 0;
    int off = 0;           // pages of segs[si] already handed out
    int64_t acc = 0;       // weight handed out so far
    for (int c = 0; c < n_ctas; ++c) {
      pl.cta_begin[c] = (int)pl.items.size();
      const int64_t goal = total_wc * (c + 1) / n_ctas;
      bool first = true;
      while (si < segs.size() && (acc < goal || c == n_ctas - 1)) {
        const Seg& sg = segs[si];
        const int64_t wpp = sg.wpp;
        if (!first) {
          if (acc + item_cost(sg) >= goal && c != n_ctas - 1) break;
          acc += item_cost(sg);
        }
        first = false;
        int64_t want = (c == n_ctas - 1) ? (sg.len - off) : (goal - acc + wpp - 1) / wpp;
        want = (want + kTilePages - 1) / kTilePages * kTilePages;
        int take = (int)std::max<int64_t>(1, std::min<int64_t>(want, sg.len - off));
        push_item(sg, off, take);
        acc += full_tiles(take) * wpp;
        off += take;
        if (off == sg.len) { ++si; off = 0; }
      }
    }
    pl.cta_begin[n_ctas] = (int)pl.items.size();
  }
  // 4b. decode-shaped calls of the four-agent decode kernel: one
  // query-side RoPE matrix per (agent tile, kv head), shared by the items
  // that split that tile's pages (the eight-slot kernel builds its own)
  if (rpa == 4 && !slots8) {
    std::map<std::pair<int32_t, int32_t>, int32_t> idx;
    for (auto& it : pl.items) {
      auto key = std::make_pair(it.agent_begin, it.head);
      auto f = idx.find(key);
      if (f == idx.end()) {
        MPair m{};
        m.head = it.head;
        m.agent_begin = it.agent_begin;
        m.n_agents = it.n_agents;
        m.row_begin = it.row_begin;
        m.zcols = rpa * it.sum_rank;
        f = idx.emplace(key, (int32_t)pl.mpairs.size()).first;
        pl.mpairs.push_back(m);
      }
      pl.item_mpair.push_back(f->second);
    }
  }
  // 5. combine lists: output row (i, c, hq) -> partial slots
  const int n_out = A * C * H_q;
  std::vector<int32_t> cnt(n_out + 1, 0);
  auto out_row = [&](const fk_work_item& it, int j) {
    int a = pl.row_agent[it.row_begin + j], cg = pl.row_cg[it.row_begin + j];
    int c = cg / G, g = cg % G;
    return (a * C + c) * H_q + it.head * G + g;
  };
  auto real = [&](const fk_work_item& it, int j) { return pl.row_agent[it.row_begin + j] >= 0; };
  for (auto& it : pl.items)
    for (int j = 0; j < it.n_rows; ++j)
      if (real(it, j)) cnt[out_row(it, j) + 1]++;
  for (int r = 0; r < n_out; ++r) {
    if (cnt[r + 1] == 0) return fail(FK_ERR_INVALID_ARG, "an output row has no keys");
    cnt[r + 1] += cnt[r];
  }
  pl.csr_ptr = cnt;
  pl.csr_slots.assign(cnt[n_out], 0);
  std::vector<int32_t> pos(cnt.begin(), cnt.end() - 1);
  for (auto& it : pl.items)
    for (int j = 0; j < it.n_rows; ++j)
      if (real(it, j)) pl.csr_slots[pos[out_row(it, j)]++] = it.partial_begin + j;
  out = std::move(pl);
  return FK_OK;
}

// Calls the chunk kernel takes: many query rows per agent and kv head.
bool use_chunk(const PoolGeom& g, int C, int compressed) {
  return !compressed && g.d == 128 && (g.H_q / g.H_kv) * C >= 128;
}

// Work list of the chunk kernel (calls with >= 128 query rows per agent
// and kv head): one item per (call agent, kv head, block of 128 of the
// agent's G*C rows, run of whole 128-token tiles).  Units are taken in the
// order (kv head, agent, row block), so that the agents reading one head's
// shared pages run side by side, and cut at tile boundaries so that each of
// at most n_ctas CTAs gets the same number of tiles.  Every item writes one
// split partial per row; the combine lists map each output row to them.
fk_status plan_chunk(int A, int C, int H_q, int H_kv, const int32_t* bt, int max_pages,
                     const int32_t* seq, int n_ctas, HostPlan& out) {
  if (A < 1 || C < 1 || H_kv < 1 || H_q % H_kv || n_ctas < 1)
    return fail(FK_ERR_INVALID_ARG, "bad call shape");
  const int G = H_q / H_kv, R = G * C, nb = (R + 127) / 128;
  for (int i = 0; i < A; ++i) {
    if (seq[i] < C) return fail(FK_ERR_INVALID_ARG, "seq_lens[i] must be >= C >= 1");
    const int np = (seq[i] + kPage - 1) / kPage;
    if (np > max_pages) return fail(FK_ERR_INVALID_ARG, "seq_len exceeds max_pages");
    for (int lp = 0; lp < np; ++lp)
      if (bt[(int64_t)i * max_pages + lp] < 0)
        return fail(FK_ERR_INVALID_ARG, "block table names no page for a live token");
  }
  int64_t total = 0;
  for (int i = 0; i < A; ++i) total += (int64_t)H_kv * nb * (((seq[i] + kPage - 1) / kPage + kTilePages - 1) / kTilePages);
  const int64_t quota = (total + n_ctas - 1) / n_ctas;
  HostPlan pl;
  pl.cta_begin.push_back(0);
  int64_t acc = 0;
  for (int h = 0; h < H_kv; ++h)
    for (int i = 0; i < A; ++i)
      for (int b = 0; b < nb; ++b) {
        const int np = (seq[i] + kPage - 1) / kPage;
        const int tiles = (np + kTilePages - 1) / kTilePages;
        int done = 0;
        while (done < tiles) {
          const int take = (int)std::min<int64_t>(tiles - done, quota - acc);
          fk_work_item it{};
          it.head = h;
          it.row_begin = 128 * b;
          it.n_rows = std::min(128, R - 128 * b);
          it.page_begin = (int)pl.pages.size();
          it.lp_begin = done * kTilePages;
          it.n_pages = std::min(take * kTilePages, np - it.lp_begin);
          it.agent_begin = i;
          it.n_agents = 1;
          it.partial_begin = pl.n_partials;
          for (int j = 0; j < it.n_pages; ++j)
            pl.pages.push_back(bt[(int64_t)i * max_pages + it.lp_begin + j]);
          pl.n_partials += it.n_rows;
          pl.items.push_back(it);
          done += take;
          acc += take;
          if (acc == quota) {
            pl.cta_begin.push_back((int)pl.items.size());
            acc = 0;
          }
        }
      }
  if (acc > 0) pl.cta_begin.push_back((int)pl.items.size());
  // combine lists: output row (i, c, hq) -> partial slots
  const int n_out = A * C * H_q;
  std::vector<int32_t> cnt(n_out + 1, 0);
  auto out_row = [&](const fk_work_item& it, int r) {
    const int ridx = it.row_begin + r, c = ridx / G, g = ridx % G;
    return (it.agent_begin * C + c) * H_q + it.head * G + g;
  };
  for (auto& it : pl.items)
    for (int r = 0; r < it.n_rows; ++r) cnt[out_row(it, r) + 1]++;
  for (int o = 0; o < n_out; ++o) {
    if (cnt[o + 1] == 0) return fail(FK_ERR_INVALID_ARG, "an output row has no keys");
    cnt[o + 1] += cnt[o];
  }
  pl.csr_ptr = cnt;
  pl.csr_slots.assign(cnt[n_out], 0);
  std::vector<int32_t> pos(cnt.begin(), cnt.end() - 1);
  for (auto& it : pl.items)
    for (int r = 0; r < it.n_rows; ++r) pl.csr_slots[pos[out_row(it, r)]++] = it.partial_begin + r;
  out = std::move(pl);
  return FK_OK;
}

// The host-side lookups of each M pair (see MPair): pool agent, padded
// rank and scale of its agents, and the q row of each query row.
void fill_mpairs(HostPlan& pl, const fk_pool* p, const int32_t* agents, int C) {
  const PoolGeom& g = p->g;
  const int G = g.H_q / g.H_kv;
  for (auto& m : pl.mpairs) {
    for (int a = 0; a < m.n_agents; ++a) {
      const int pa = agents[pl.tile_agents[m.agent_begin + a]];
      m.pool_agent[a] = pa;
      m.rp[a] = p->agents[pa].rp;
      m.s[a] = p->agents[pa].s;
    }
    for (int row = 0; row < m.n_agents * 4; ++row) {
      const int ci = pl.row_agent[m.row_begin + row], cg = pl.row_cg[m.row_begin + row];
      m.qrow[row] = (ci * C + cg / G) * g.H_q + m.head * G + cg % G;
    }
  }
}

// The four-agent decode kernel's item records (see DecItem): the lookups
// of each item's agents, rows and first pages, in CTA order.
std::vector<DecItem> make_ditems(const HostPlan& pl, const fk_pool* p, const int32_t* agents,
                                 const int32_t* seq, int C, int causal) {
  const PoolGeom& g = p->g;
  const int G = g.H_q / g.H_kv;
  auto rec = [&](int it) {
    const fk_work_item& w = pl.items[it];
    DecItem d{};
    d.head = w.head;
    d.n_rows = w.n_rows;
    d.n_pages = w.n_pages;
    d.lp_begin = w.lp_begin;
    d.n_ag = w.n_agents;
    d.partial_begin = w.partial_begin;
    d.page_begin = w.page_begin;
    d.next = -1;
    d.mbytes = it;           // item index until pack_plan places the M matrices
    int col = 0, lvc = 0;
    for (int a = 0; a < kMaxAgentsPerTile; ++a) {
      d.col[a] = col;
      d.qrow[4 * a] = d.qrow[4 * a + 1] = d.qrow[4 * a + 2] = d.qrow[4 * a + 3] = -1;
      if (a >= w.n_agents) continue;
      const int pa = agents[pl.tile_agents[w.agent_begin + a]];
      d.pool_agent[a] = pa;
      d.rp[a] = p->agents[pa].rp;
      d.s[a] = p->agents[pa].s;
      d.rc_off[a] = p->agents[pa].rc_off;
      col += d.rp[a];
      // Shared-A: an agent reading the same residual rows as an earlier one
      // uses that agent's block of the Lv^T stage
      int share = -1;
      for (int b = 0; b < a && share < 0; ++b)
        if (d.rc_off[b] == d.rc_off[a]) share = b;
      d.lvcol[a] = share >= 0 ? d.lvcol[share] : lvc;
      if (share < 0) lvc += d.rp[a];
    }
    d.sum_rp = col;
    d.lv_rp = lvc;
    // at most two agents leave the second compute warpgroup without rows;
    // with six or more rank groups it takes half of them
    d.split = (w.n_agents <= 2 && col >= 48) ? 1 : 0;
    for (int j = 0; j < 4 * kMaxAgentsPerTile; ++j) {
      d.row_lim[j] = 0;
      if (j >= w.n_rows) continue;
      const int ci = pl.row_agent[w.row_begin + j], cg = pl.row_cg[w.row_begin + j];
      if (ci < 0) continue;
      d.qrow[j] = (ci * C + cg / G) * g.H_q + w.head * G + cg % G;
      const int T = seq[ci];
      d.row_lim[j] = causal ? std::min(T, T - C + cg / G + 1) : T;
    }
    for (int h = 0; h < 2; ++h) {
      int mn = 0x7fffffff;
      for (int j = 8 * h; j < 8 * h + 8; ++j) mn = std::min(mn, j < w.n_rows ? d.row_lim[j] : 0);
      d.lim_min[h] = mn;
    }
    for (int k = 0; k < kTilePages; ++k)
      d.first_pages[k] = k < w.n_pages ? pl.pages[w.page_begin + k] : 0;
    return d;
  };
  const int n_ctas = (int)pl.cta_begin.size() - 1;
  std::vector<DecItem> out(n_ctas);
  for (int c = 0; c < n_ctas; ++c) {
    const int b = pl.cta_begin[c], e = pl.cta_begin[c + 1];
    if (b == e) {
      out[c] = DecItem{};
      out[c].next = -1;
      continue;
    }
    out[c] = rec(b);
    int prev = c;
    for (int it = b + 1; it < e; ++it) {
      out[prev].next = (int)out.size();
      prev = (int)out.size();
      out.push_back(rec(it));
    }
  }
  return out;
}

// Pack a work list into the workspace image: the plan arrays, then the
// split partials, then the four-agent decode kernel's M matrices.  Returns
// the bytes of workspace the call needs (blob covers the plan arrays only).
int64_t pack_plan(const HostPlan& pl, int A, int C, int causal, const int32_t* agents,
                  const int32_t* seq, const PoolGeom& g, const std::vector<DecItem>& ditems,
                  std::vector<uint8_t>& blob, PlanDev& pd) {
  pd = PlanDev{};
  pd.n_items = (int)pl.items.size();
  pd.n_rows = (int)pl.row_agent.size();
  pd.n_pages = (int)pl.pages.size();
  pd.n_tile_agents = (int)pl.tile_agents.size();
  pd.A = A; pd.C = C; pd.causal = causal ? 1 : 0;
  pd.n_out_rows = A * C * g.H_q;
  pd.n_partials = pl.n_partials;
  pd.partial_stride = g.d + g.rmax_pad + 4;
  blob.clear();
  auto put = [&](const void* src, size_t bytes) {
    int64_t o = align_up((int64_t)blob.size(), 256);
    blob.resize(o + bytes);
    if (bytes) std::memcpy(blob.data() + o, src, bytes);
    return o;
  };
  std::vector<CallAgent> ca(A);
  for (int i = 0; i < A; ++i) ca[i] = CallAgent{agents[i], seq[i]};
  pd.off_items = put(pl.items.data(), pl.items.size() * sizeof(fk_work_item));
  pd.off_row_agent = put(pl.row_agent.data(), pl.row_agent.size() * 4);
  pd.off_row_cg = put(pl.row_cg.data(), pl.row_cg.size() * 4);
  pd.off_pages = put(pl.pages.data(), pl.pages.size() * 4);
  pd.off_tile_agents = put(pl.tile_agents.data(), pl.tile_agents.size() * 4);
  pd.off_call_agents = put(ca.data(), ca.size() * sizeof(CallAgent));
  pd.off_csr_ptr = put(pl.csr_ptr.data(), pl.csr_ptr.size() * 4);
  pd.off_csr_slots = put(pl.csr_slots.data(), pl.csr_slots.size() * 4);
  pd.off_cta = put(pl.cta_begin.data(), pl.cta_begin.size() * 4);
  pd.n_ctas = (int)pl.cta_begin.size() - 1;
  // M offsets are known only once the partials are placed: reserve the
  // pair table and the item records, fill them in below
  std::vector<MPair> mp = pl.mpairs;
  std::vector<DecItem> di = ditems;
  pd.n_mpairs = (int)mp.size();
  pd.off_mpairs = put(mp.data(), mp.size() * sizeof(MPair));
  pd.n_ditems = (int)di.size();
  pd.off_ditems = put(di.data(), di.size() * sizeof(DecItem));
  pd.off_partials = align_up((int64_t)blob.size(), 256);
  int64_t need = pd.off_partials + (int64_t)pd.n_partials * pd.partial_stride * 4;
  need = align_up(need, 1024);
  for (auto& m : mp) {
    m.mofs = need;
    need += align_up((int64_t)m.zcols * g.d * 2, 1024);
  }
  if (!mp.empty()) std::memcpy(blob.data() + pd.off_mpairs, mp.data(), mp.size() * sizeof(MPair));
  for (auto& d : di) {
    if (d.n_pages == 0) continue;
    const MPair& m = mp[pl.item_mpair[d.mbytes]];
    d.mofs = m.mofs;
    d.mbytes = m.zcols * g.d * 2;
  }
  if (!di.empty()) std::memcpy(blob.data() + pd.off_ditems, di.data(), di.size() * sizeof(DecItem));
  return need;
}

// Which kernel a call runs, and its work list packed for the workspace:
// calls with many rows per agent and kv head take the chunk kernel;
// decode-shaped calls (four rows per agent) with d = 128 on the
// uncompressed pool take the eight-slot decode kernel when the pool was
// created with it; the rest the four-agent decode kernel or the general
// kernel.
fk_status build_call_plan(const fk_pool* p, const int32_t* agents, const int32_t* bt, int max_pages,
                          const int32_t* seq, const int32_t* rp, int A, int C, int causal,
                          int compressed, HostPlan& pl, std::vector<uint8_t>& blob, PlanDev& pd,
                          int64_t& need) {
  const PoolGeom& g = p->g;
  const bool chunk = use_chunk(g, C, compressed);
  const bool dec8 = p->slots8 && !chunk && !compressed && g.d == 128 && g.G * C == 4;
  fk_status s = chunk ? plan_chunk(A, C, g.H_q, g.H_kv, bt, max_pages, seq, p->num_sms, pl)
              : dec8  ? plan_build(A, C, g.H_q, g.H_kv, kPage, bt, max_pages, seq, rp,
                                   4 * kDecodeSlots, 2 * kDecodeHalfRank, p->num_sms, pl, true)
                      : plan_build(A, C, g.H_q, g.H_kv, kPage, bt, max_pages, seq, rp, kMaxRows,
                                   kMaxRankSum, p->num_sms, pl);
  if (s != FK_OK) return s;
  // the four-agent decode kernel reads its items as flat records
  std::vector<DecItem> ditems;
  if (!chunk && !dec8 && g.G * C == 4 && (g.d == 64 || g.d == 128)) {
    fill_mpairs(pl, p, agents, C);
    ditems = make_ditems(pl, p, agents, seq, C, causal);
  }
  need = pack_plan(pl, A, C, causal, agents, seq, g, ditems, blob, pd);
  pd.chunk = chunk ? 1 : 0;
  pd.slots8 = dec8 ? 1 : 0;
  return FK_OK;
}

}  // namespace

// Work list of fk_residual_attention_noalloc, kept apart from the pool's own
// cache: the static scratch is shared by every pool of the process, one
// entry per device.  Entries are keyed by the pool's uid, which no later
// pool reuses (a new pool may get a freed pool's address), and a destroyed
// pool's entries are cleared.  The uploaded blob stays here: its host
// memory outlives the copy.
namespace {
struct NoallocCache {
  uint64_t pool_uid = 0;
  std::vector<int32_t> key;
  std::vector<uint8_t> blob;
  PlanDev pd{};
};
NoallocCache g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;
std::atomic<uint64_t> g_next_pool_uid{1};
}  // namespace

// ================================================================= ABI ==

// Last-error text for the other translation units of the library.
void fk_internal_set_error(const char* msg) { g_err = msg; }

extern "C" {

const char* fk_last_error(void) { return g_err.c_str(); }

const char* fk_version(void) { return "forkkv-gb300 0.1 (sm_103a)"; }

size_t fk_pool_bytes(const fk_pool_config* cfg) {
  if (validate_config(cfg) != FK_OK) return 0;
  return (size_t)total_bytes(make_geom(cfg));
}

fk_status fk_pool_create(const fk_pool_config* cfg, void* dev_buf, size_t bytes,
                         fk_pool** out) {
  fk_status st = validate_config(cfg);
  if (st != FK_OK) return st;
  if (!out) return fail(FK_ERR_INVALID_ARG, "out is NULL");
  if (!dev_buf || ((uintptr_t)dev_buf % 256))
    return fail(FK_ERR_INVALID_ARG, "dev_buf must be a 256-byte aligned device pointer");
  PoolGeom g = make_geom(cfg);
  if ((int64_t)bytes < total_bytes(g))
    return fail(FK_ERR_INVALID_ARG, "dev_buf smaller than fk_pool_bytes(cfg)");
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, dev_buf);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return fail(FK_ERR_INVALID_ARG, "dev_buf is not device memory");
  }
  fk_pool* p = new fk_pool();
  p->uid = g_next_pool_uid.fetch_add(1);
  p->cfg = *cfg;
  p->g = g;
  p->g.base = (uint8_t*)dev_buf;
  cudaGetDevice(&p->device);
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  {
    const char* ds = std::getenv("FORKKV_DECODE_SLOTS");
    p->slots8 = ds != nullptr && std::strcmp(ds, "8") == 0;
  }
  p->refcount.assign(g.num_pages, 0);
  p->free_list.reserve(g.num_pages);
  for (int i = g.num_pages - 1; i >= 0; --i) p->free_list.push_back(i);
  p->fill.assign((size_t)g.L * g.num_pages, 0);
  p->agents.assign(g.max_agents, {});
  p->rc_free[rc_arena_offset(g)] = rc_arena_bytes(g);
  e = cudaEventCreateWithFlags(&p->stage.done, cudaEventDisableTiming);
  if (e != cudaSuccess) { delete p; return cuda_fail(e, "cudaEventCreate"); }
  // zero the small tables (agents, error word); write the RoPE table:
  // theta_i in fp32 plus its fp32 residual, and the exact rotation by one
  // 128-token tile, all computed in double.
  // zero the page stores (rows never appended must read as finite zeros),
  // the small tables and the compressed copy
  e = cudaMemset(p->g.base + g.off_kb, 0, 2 * g.kb_layer_bytes * g.L);
  if (e == cudaSuccess) e = cudaMemset(p->g.base + g.off_agents, 0, g.off_lvmap + 128LL * g.max_agents - g.off_agents);
  if (e == cudaSuccess && g.compressed)
    e = cudaMemset(p->g.base + g.off_kq, 0, g.off_kmax + 4LL * g.L - g.off_kq);
  if (e != cudaSuccess) { cudaEventDestroy(p->stage.done); delete p; return cuda_fail(e, "cudaMemset"); }
  // RoPE table: theta_i as fp32, then theta_i / (2 pi) as a 64-bit binary
  // fraction so that kernels reduce t * theta_i modulo 2 pi exactly with an
  // integer multiply.
  std::vector<uint8_t> rope(64 * 4 + 64 * 8, 0);
  for (int i = 0; i < g.d / 2; ++i) {
    long double th = std::pow((long double)g.rope_base, -2.0L * i / g.d);
    float f = (float)th;
    std::memcpy(rope.data() + 4 * i, &f, 4);
    long double frac = th / (2.0L * 3.14159265358979323846264338327950288L);
    unsigned long long fx = (unsigned long long)std::ldexp(frac, 64);
    std::memcpy(rope.data() + 256 + 8 * i, &fx, 8);
  }
  e = cudaMemcpy(p->g.base + g.off_rope, rope.data(), rope.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) { cudaEventDestroy(p->stage.done); delete p; return cuda_fail(e, "cudaMemcpy"); }
  // per-position rotations (from the fractions above), complete before the
  // call returns
  if (g.off_trig >= 0) {
    e = (cudaError_t)launch_trig_table(p->g);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) { cudaEventDestroy(p->stage.done); delete p; return cuda_fail(e, "RoPE table"); }
  }
  *out = p;
  return FK_OK;
}

fk_status fk_pool_destroy(fk_pool* p) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (NoallocCache& c : g_noalloc)
      if (c.pool_uid == p->uid) c = NoallocCache();
  }
  if (p->stage.pending) cudaEventSynchronize(p->stage.done);
  if (p->stage.host) cudaFreeHost(p->stage.host);
  if (p->stage.done) cudaEventDestroy(p->stage.done);
  delete p;
  return FK_OK;
}

fk_status fk_pool_region(const fk_pool* p, int region, size_t* offset, size_t* bytes) {
  if (!p || !offset || !bytes) return fail(FK_ERR_INVALID_ARG, "NULL argument");
  const PoolGeom& g = p->g;
  int64_t tok = (int64_t)g.L * g.num_pages * g.H_kv * kPage;
  int64_t o = -1, b = 0;
  switch (region) {
    case FK_REGION_KB: o = g.off_kb; b = g.kb_layer_bytes * g.L; break;
    case FK_REGION_VB: o = g.off_vb; b = g.kb_layer_bytes * g.L; break;
    case FK_REGION_RC: o = rc_arena_offset(g); b = rc_arena_bytes(g); break;
    case FK_REGION_KQ: o = g.off_kq; b = tok * g.d; break;
    case FK_REGION_VC: o = g.off_vc; b = tok * (3 * g.d / 8); break;
    case FK_REGION_VN: o = g.off_vn; b = tok * 4; break;
    case FK_REGION_KS: o = g.off_ks; b = 4LL * g.L; break;
    default: return fail(FK_ERR_INVALID_ARG, "unknown region");
  }
  if (o < 0) return fail(FK_ERR_INVALID_ARG, "region absent (pool not compressed)");
  *offset = (size_t)o;
  *bytes = (size_t)b;
  return FK_OK;
}

fk_status fk_pages_alloc(fk_pool* p, int n, int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return fail(FK_ERR_INVALID_ARG, "bad arguments");
  if ((size_t)n > p->free_list.size())
    return fail(FK_ERR_OUT_OF_PAGES, "not enough free pages");
  for (int i = 0; i < n; ++i) {
    int32_t id = p->free_list.back();
    p->free_list.pop_back();
    p->refcount[id] = 1;
    for (int l = 0; l < p->g.L; ++l) p->fill[(size_t)l * p->g.num_pages + id] = 0;
    ids[i] = id;
  }
  return FK_OK;
}

fk_status fk_pages_release(fk_pool* p, int n, const int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return fail(FK_ERR_INVALID_ARG, "bad arguments");
  std::map<int32_t, int> drops;
  for (int i = 0; i < n; ++i) {
    if (ids[i] == -1) continue;
    if (ids[i] < 0 || ids[i] >= p->g.num_pages) return fail(FK_ERR_INVALID_ARG, "page id out of range");
    drops[ids[i]]++;
  }
  for (auto& kv : drops)
    if (p->refcount[kv.first] < kv.second)
      return fail(FK_ERR_INVALID_ARG, "releasing a page that is already free");
  for (auto& kv : drops) {
    p->refcount[kv.first] -= kv.second;
    if (p->refcount[kv.first] == 0) p->free_list.push_back(kv.first);
  }
  p->plan_valid = false;
  ++p->plan_gen;
  return FK_OK;
}

fk_status fk_fork(fk_pool* p, const int32_t* parent, int n, int32_t* child) {
  if (!p || n < 0 || (n > 0 && (!parent || !child))) return fail(FK_ERR_INVALID_ARG, "bad arguments");
  for (int i = 0; i < n; ++i) {
    if (parent[i] == -1) continue;
    if (parent[i] < 0 || parent[i] >= p->g.num_pages || p->refcount[parent[i]] <= 0)
      return fail(FK_ERR_INVALID_ARG, "parent row names a free or invalid page");
  }
  for (int i = 0; i < n; ++i) {
    child[i] = parent[i];
    if (parent[i] >= 0) p->refcount[parent[i]]++;
  }
  return FK_OK;
}

int fk_page_refcount(const fk_pool* p, int32_t id) {
  if (!p || id < 0 || id >= p->g.num_pages) return -1;
  return p->refcount[id];
}

fk_status fk_agent_register(fk_pool* p, int agent, int rank, float s,
                            const uint16_t* Bk, const uint16_t* Bv, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (agent < 0 || agent >= p->g.max_agents) return fail(FK_ERR_INVALID_ARG, "agent id out of range");
  if (p->agents[agent].live) return fail(FK_ERR_INVALID_ARG, "agent id already registered");
  if (rank < 8 || rank % 8 || rank > p->cfg.max_rank)
    return fail(FK_ERR_INVALID_ARG, "rank must be a multiple of 8 and <= max_rank");
  if (!Bk || !Bv) return fail(FK_ERR_INVALID_ARG, "Bk/Bv are NULL");
  if (!std::isfinite(s)) return fail(FK_ERR_INVALID_ARG, "s must be finite");
  int rp = rank_pad(rank);
  int64_t need = (int64_t)p->g.L * rc_layer_bytes(p->g, rp);
  auto it = p->rc_free.begin();
  for (; it != p->rc_free.end(); ++it)
    if (it->second >= need) break;
  if (it == p->rc_free.end()) return fail(FK_ERR_OOM, "rCache arena full");
  int64_t off = it->first, len = it->second;
  p->rc_free.erase(it);
  if (len > need) p->rc_free[off + need] = len - need;
  auto& A = p->agents[agent];
  A.live = true; A.rank = rank; A.rp = rp; A.s = s; A.rc_off = off; A.rc_bytes = need;
  p->rc_users[off] = 1;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(p->g.base + off, 0, need, st);
  AgentDev dv{rp, s, off};
  if (e == cudaSuccess)
    e = (cudaError_t)launch_agent_register(p->g, agent, rank, rp, dv, Bk, Bv, stream);
  fk_status r2 = (e == cudaSuccess) ? upload_agent(p, agent, st) : cuda_fail(e, "agent register");
  if (r2 != FK_OK) {
    A = fk_pool::Agent{};
    p->rc_users.erase(off);
    p->rc_free[off] = need;
    return r2;
  }
  p->plan_valid = false;
  ++p->plan_gen;
  return FK_OK;
}

fk_status fk_agent_register_shared(fk_pool* p, int agent, int src, float s, const uint16_t* Bk,
                                   const uint16_t* Bv, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (agent < 0 || agent >= p->g.max_agents || src < 0 || src >= p->g.max_agents)
    return fail(FK_ERR_INVALID_ARG, "agent id out of range");
  if (p->agents[agent].live) return fail(FK_ERR_INVALID_ARG, "agent id already registered");
  if (!p->agents[src].live) return fail(FK_ERR_INVALID_ARG, "source agent is not registered");
  if (!Bk || !Bv) return fail(FK_ERR_INVALID_ARG, "Bk/Bv are NULL");
  if (!std::isfinite(s)) return fail(FK_ERR_INVALID_ARG, "s must be finite");
  const auto S = p->agents[src];
  auto& A = p->agents[agent];
  A.live = true; A.rank = S.rank; A.rp = S.rp; A.s = s; A.rc_off = S.rc_off; A.rc_bytes = S.rc_bytes;
  cudaStream_t st = (cudaStream_t)stream;
  AgentDev dv{A.rp, s, A.rc_off};
  cudaError_t e = (cudaError_t)launch_agent_register(p->g, agent, A.rank, A.rp, dv, Bk, Bv, stream);
  fk_status r2 = (e == cudaSuccess) ? upload_agent(p, agent, st) : cuda_fail(e, "agent register");
  if (r2 != FK_OK) {
    A = fk_pool::Agent{};
    return r2;
  }
  ++p->rc_users[A.rc_off];
  p->plan_valid = false;
  ++p->plan_gen;
  return FK_OK;
}

fk_status fk_agent_release(fk_pool* p, int agent) {
  if (!p || agent < 0 || agent >= p->g.max_agents || !p->agents[agent].live)
    return fail(FK_ERR_INVALID_ARG, "agent not registered");
  auto& A = p->agents[agent];
  // rows still read by another agent (Shared-A) stay
  auto u = p->rc_users.find(A.rc_off);
  if (u != p->rc_users.end() && u->second > 1) {
    --u->second;
    A = fk_pool::Agent{};
    p->plan_valid = false;
    ++p->plan_gen;
    return upload_agent(p, agent, nullptr);
  }
  if (u != p->rc_users.end()) p->rc_users.erase(u);
  // return the range and merge neighbours
  int64_t off = A.rc_off, len = A.rc_bytes;
  auto nx = p->rc_free.lower_bound(off);
  if (nx != p->rc_free.end() && nx->first == off + len) { len += nx->second; p->rc_free.erase(nx); }
  auto pv = p->rc_free.lower_bound(off);
  if (pv != p->rc_free.begin()) {
    --pv;
    if (pv->first + pv->second == off) { off = pv->first; len += pv->second; p->rc_free.erase(pv); }
  }
  p->rc_free[off] = len;
  A = fk_pool::Agent{};
  p->plan_valid = false;
  ++p->plan_gen;
  return upload_agent(p, agent, nullptr);
}

fk_status fk_agent_rcache(const fk_pool* p, int agent, size_t* lk_offset, size_t* layer_bytes,
                          int* padded_rank) {
  if (!p || !lk_offset || !layer_bytes || !padded_rank) return fail(FK_ERR_INVALID_ARG, "NULL argument");
  if (agent < 0 || agent >= p->g.max_agents || !p->agents[agent].live)
    return fail(FK_ERR_INVALID_ARG, "agent not registered");
  const auto& A = p->agents[agent];
  *lk_offset = (size_t)A.rc_off;
  *layer_bytes = (size_t)rc_layer_bytes(p->g, A.rp);
  *padded_rank = A.rp;
  return FK_OK;
}

fk_status fk_base_append(fk_pool* p, int layer, int32_t* row, int max_pages, int pos,
                         int n, const uint16_t* Kb, const uint16_t* Vb, void* stream) {
  if (!p || !row) return fail(FK_ERR_INVALID_ARG, "NULL argument");
  if (layer < 0 || layer >= p->g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (pos < 0 || n < 0) return fail(FK_ERR_INVALID_ARG, "negative position or count");
  if (n == 0) return FK_OK;
  if (!Kb || !Vb) return fail(FK_ERR_INVALID_ARG, "Kb/Vb are NULL");
  int lp0 = pos / kPage, lp1 = (pos + n - 1) / kPage;
  if (lp1 >= max_pages) return fail(FK_ERR_INVALID_ARG, "append runs past max_pages");
  for (int lp = lp0; lp <= lp1; ++lp)
    if (row[lp] < -1 || row[lp] >= p->g.num_pages || (row[lp] >= 0 && p->refcount[row[lp]] <= 0))
      return fail(FK_ERR_INVALID_ARG, "block table row names a free or invalid page");
  int need_new = 0;
  for (int lp = lp0; lp <= lp1; ++lp)
    if (row[lp] < 0 || p->refcount[row[lp]] > 1) need_new++;
  if ((size_t)need_new > p->free_list.size())
    return fail(FK_ERR_OUT_OF_PAGES, "not enough free pages for append / copy-on-write");
  cudaStream_t st = (cudaStream_t)stream;
  const PoolGeom& g = p->g;
  for (int lp = lp0; lp <= lp1; ++lp) {
    if (row[lp] < 0) {
      int32_t id;
      fk_pages_alloc(p, 1, &id);
      row[lp] = id;
    } else if (p->refcount[row[lp]] > 1) {
      // copy-on-write: never write a page other rows still name
      int32_t old = row[lp], id;
      fk_pages_alloc(p, 1, &id);
      int64_t blk = (int64_t)g.H_kv * g.page_bytes;
      for (int64_t region : {g.off_kb, g.off_vb}) {
        cudaError_t e = cudaMemcpy2DAsync(g.base + region + id * blk, g.kb_layer_bytes,
                                          g.base + region + old * blk, g.kb_layer_bytes,
                                          blk, g.L, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "copy-on-write copy");
      }
      if (g.compressed) {
        int64_t tokb = (int64_t)g.H_kv * kPage;
        struct R { int64_t off, per_tok; } regs[3] = {{g.off_kq, g.d}, {g.off_vc, 3 * g.d / 8}, {g.off_vn, 4}};
        for (auto& r : regs) {
          int64_t b = tokb * r.per_tok;
          cudaError_t e = cudaMemcpy2DAsync(g.base + r.off + id * b, b * g.num_pages,
                                            g.base + r.off + old * b, b * g.num_pages, b, g.L,
                                            cudaMemcpyDeviceToDevice, st);
          if (e != cudaSuccess) return cuda_fail(e, "copy-on-write copy");
        }
      }
      for (int l = 0; l < g.L; ++l)
        p->fill[(size_t)l * g.num_pages + id] = p->fill[(size_t)l * g.num_pages + old];
      p->refcount[old]--;
      row[lp] = id;
    }
  }
  // write in launches of at most 64 pages
  for (int c0 = lp0; c0 <= lp1; c0 += 64) {
    int c1 = std::min(lp1, c0 + 63);
    int t0 = std::max(pos, c0 * kPage), t1 = std::min(pos + n, (c1 + 1) * kPage);
    int e = launch_base_append(g, layer, row + c0, c1 - c0 + 1, t0, t1 - t0,
                               Kb + (int64_t)(t0 - pos) * g.H_kv * g.d,
                               Vb + (int64_t)(t0 - pos) * g.H_kv * g.d, stream);
    if (e != 0) return cuda_fail((cudaError_t)e, "base append kernel");
  }
  for (int lp = lp0; lp <= lp1; ++lp) {
    int end = std::min(pos + n - lp * kPage, kPage);
    uint8_t& f = p->fill[(size_t)layer * g.num_pages + row[lp]];
    f = (uint8_t)std::max<int>(f, end);
  }
  p->plan_valid = false;
  ++p->plan_gen;
  return FK_OK;
}

fk_status fk_residual_append(fk_pool* p, int layer, int agent, int pos, int n,
                             const uint16_t* Lk, const uint16_t* Lv, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (layer < 0 || layer >= p->g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (agent < 0 || agent >= p->g.max_agents || !p->agents[agent].live)
    return fail(FK_ERR_INVALID_ARG, "agent not registered");
  if (pos < 0 || n < 0 || (int64_t)pos + n > p->cfg.max_tokens)
    return fail(FK_ERR_INVALID_ARG, "rows out of the rCache capacity");
  if (n == 0) return FK_OK;
  if (!Lk || !Lv) return fail(FK_ERR_INVALID_ARG, "Lk/Lv are NULL");
  const auto& A = p->agents[agent];
  AgentDev dv{A.rp, A.s, A.rc_off};
  int e = launch_residual_append(p->g, layer, dv, A.rank, pos, n, Lk, Lv, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "residual append kernel");
  return FK_OK;
}

fk_status fk_residual_prefill(fk_pool* p, int layer, int agent, int pos, int n,
                              const uint16_t* X, const uint16_t* Ak, const uint16_t* Av,
                              int d_model, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (layer < 0 || layer >= p->g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (agent < 0 || agent >= p->g.max_agents || !p->agents[agent].live)
    return fail(FK_ERR_INVALID_ARG, "agent not registered");
  if (pos < 0 || n < 0 || (int64_t)pos + n > p->cfg.max_tokens)
    return fail(FK_ERR_INVALID_ARG, "rows out of the rCache capacity");
  if (d_model <= 0 || d_model % 128 != 0)
    return fail(FK_ERR_INVALID_ARG, "d_model must be a positive multiple of 128");
  if (n == 0) return FK_OK;
  if (!X || !Ak || !Av) return fail(FK_ERR_INVALID_ARG, "X/Ak/Av are NULL");
  if (((uintptr_t)X | (uintptr_t)Ak | (uintptr_t)Av) % 16 != 0)
    return fail(FK_ERR_INVALID_ARG, "X/Ak/Av must be 16-byte aligned");
  const auto& A = p->agents[agent];
  // X as 128-row x 64-feature boxes in the 128-byte swizzle the MMA reads;
  // rows past n are filled with zeros
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return fail(FK_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  alignas(64) CUtensorMap xm;
  const cuuint64_t dims[2] = {(cuuint64_t)d_model, (cuuint64_t)n};
  const cuuint64_t strides[1] = {(cuuint64_t)d_model * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)X, dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return fail(FK_ERR_CUDA, "cuTensorMapEncodeTiled failed for X");
  AgentDev dv{A.rp, A.s, A.rc_off};
  int e = launch_residual_prefill(p->g, layer, dv, A.rank, pos, n, d_model, &xm, Ak, Av, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "residual prefill kernel");
  return FK_OK;
}

fk_status fk_pool_compress(fk_pool* p, int layer, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (!p->g.compressed) return fail(FK_ERR_INVALID_ARG, "pool has no compressed copy");
  if (layer < 0 || layer >= p->g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  std::vector<int32_t> ids, fills;
  for (int id = 0; id < p->g.num_pages; ++id) {
    int f = p->fill[(size_t)layer * p->g.num_pages + id];
    if (p->refcount[id] > 0 && f > 0) { ids.push_back(id); fills.push_back(f); }
  }
  const int n = (int)ids.size();
  std::vector<int32_t> buf(2 * (size_t)n);
  std::copy(ids.begin(), ids.end(), buf.begin());
  std::copy(fills.begin(), fills.end(), buf.begin() + n);
  if ((int64_t)buf.size() * 4 > p->g.meta_bytes) return fail(FK_ERR_OOM, "meta region too small");
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* d = (int32_t*)(p->g.base + p->g.off_meta);
  if (n > 0) {
    fk_status s = stage_upload(p, buf.data(), buf.size() * 4, d, st);
    if (s != FK_OK) return s;
  }
  int e = launch_compress(p->g, layer, d, d + n, n, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "compress kernels");
  return FK_OK;
}

fk_status fk_pool_load_compressed(fk_pool* p, int layer, const int32_t* ids, int n,
                                  const int8_t* kq, const uint8_t* vc, const float* vn,
                                  float k_scale, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  if (!p->g.compressed) return fail(FK_ERR_INVALID_ARG, "pool has no compressed copy");
  if (layer < 0 || layer >= p->g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (n < 0 || (n > 0 && (!ids || !kq || !vc || !vn))) return fail(FK_ERR_INVALID_ARG, "bad arguments");
  if (!(k_scale > 0.f) || !std::isfinite(k_scale)) return fail(FK_ERR_INVALID_ARG, "k_scale must be > 0");
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->g.num_pages) return fail(FK_ERR_INVALID_ARG, "page id out of range");
  if ((int64_t)n * 4 > p->g.meta_bytes) return fail(FK_ERR_OOM, "meta region too small");
  cudaStream_t st = (cudaStream_t)stream;
  int32_t* d = (int32_t*)(p->g.base + p->g.off_meta);
  if (n > 0) {
    fk_status s = stage_upload(p, ids, (size_t)n * 4, d, st);
    if (s != FK_OK) return s;
  }
  int e = launch_load_compressed(p->g, layer, d, n, kq, vc, vn, k_scale, stream);
  if (e != 0) return cuda_fail((cudaError_t)e, "load compressed kernel");
  return FK_OK;
}

fk_status fk_plan_host(int A, int C, int H_q, int H_kv, int page_size,
                       const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                       const int32_t* ranks, int max_rows, int max_rank_sum, int target_items,
                       fk_work_item* items, int cap_items, int* n_items,
                       int32_t* row_agent, int32_t* row_cg, int cap_rows, int* n_rows,
                       int32_t* page_ids, int cap_pages, int* n_pages,
                       int32_t* tile_agents, int cap_tile_agents, int* n_tile_agents) {
  if (page_size != kPage) return fail(FK_ERR_UNSUPPORTED, "page_size must be 16");
  if (!ranks) return fail(FK_ERR_INVALID_ARG, "ranks is NULL");
  std::vector<int32_t> rp(A > 0 ? A : 0);
  for (int i = 0; i < A; ++i) rp[i] = rank_pad(ranks[i]);
  HostPlan pl;
  fk_status s = plan_build(A, C, H_q, H_kv, page_size, block_table, max_pages, seq_lens,
                           rp.data(), max_rows, max_rank_sum, target_items, pl);
  if (s != FK_OK) return s;
  if (n_items) *n_items = (int)pl.items.size();
  if (n_rows) *n_rows = (int)pl.row_agent.size();
  if (n_pages) *n_pages = (int)pl.pages.size();
  if (n_tile_agents) *n_tile_agents = (int)pl.tile_agents.size();
  if ((int)pl.items.size() > cap_items || (int)pl.row_agent.size() > cap_rows ||
      (int)pl.pages.size() > cap_pages || (int)pl.tile_agents.size() > cap_tile_agents)
    return fail(FK_ERR_OOM, "output capacity too small");
  if (items) std::copy(pl.items.begin(), pl.items.end(), items);
  if (row_agent) std::copy(pl.row_agent.begin(), pl.row_agent.end(), row_agent);
  if (row_cg) std::copy(pl.row_cg.begin(), pl.row_cg.end(), row_cg);
  if (page_ids) std::copy(pl.pages.begin(), pl.pages.end(), page_ids);
  if (tile_agents) std::copy(pl.tile_agents.begin(), pl.tile_agents.end(), tile_agents);
  return FK_OK;
}

fk_status fk_plan_host_slots8(int A, int C, int H_q, int H_kv, int page_size,
                              const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                              const int32_t* ranks, int target_items, fk_work_item* items,
                              int cap_items, int* n_items, int32_t* row_agent, int32_t* row_cg,
                              int cap_rows, int* n_rows, int32_t* page_ids, int cap_pages,
                              int* n_pages, int32_t* tile_agents, int cap_tile_agents,
                              int* n_tile_agents) {
  if (page_size != kPage) return fail(FK_ERR_UNSUPPORTED, "page_size must be 16");
  if (!ranks) return fail(FK_ERR_INVALID_ARG, "ranks is NULL");
  std::vector<int32_t> rp(A > 0 ? A : 0);
  for (int i = 0; i < A; ++i) rp[i] = rank_pad(ranks[i]);
  HostPlan pl;
  fk_status s = plan_build(A, C, H_q, H_kv, page_size, block_table, max_pages, seq_lens,
                           rp.data(), 4 * kDecodeSlots, 2 * kDecodeHalfRank, target_items, pl, true);
  if (s != FK_OK) return s;
  if (n_items) *n_items = (int)pl.items.size();
  if (n_rows) *n_rows = (int)pl.row_agent.size();
  if (n_pages) *n_pages = (int)pl.pages.size();
  if (n_tile_agents) *n_tile_agents = (int)pl.tile_agents.size();
  if ((int)pl.items.size() > cap_items || (int)pl.row_agent.size() > cap_rows ||
      (int)pl.pages.size() > cap_pages || (int)pl.tile_agents.size() > cap_tile_agents)
    return fail(FK_ERR_OOM, "output capacity too small");
  if (items) std::copy(pl.items.begin(), pl.items.end(), items);
  if (row_agent) std::copy(pl.row_agent.begin(), pl.row_agent.end(), row_agent);
  if (row_cg) std::copy(pl.row_cg.begin(), pl.row_cg.end(), row_cg);
  if (page_ids) std::copy(pl.pages.begin(), pl.pages.end(), page_ids);
  if (tile_agents) std::copy(pl.tile_agents.begin(), pl.tile_agents.end(), tile_agents);
  return FK_OK;
}

fk_status fk_plan_chunk_host(int A, int C, int H_q, int H_kv, const int32_t* block_table,
                            int max_pages, const int32_t* seq_lens, int n_ctas,
                            fk_work_item* items, int cap_items, int* n_items, int32_t* cta_begin,
                            int cap_cta, int* n_cta, int32_t* page_ids, int cap_pages,
                            int* n_pages, int32_t* csr_ptr, int cap_ptr, int32_t* csr_slots,
                            int cap_slots, int* n_slots) {
  if (!block_table || !seq_lens) return fail(FK_ERR_INVALID_ARG, "NULL table");
  HostPlan pl;
  fk_status s = plan_chunk(A, C, H_q, H_kv, block_table, max_pages, seq_lens, n_ctas, pl);
  if (s != FK_OK) return s;
  if (n_items) *n_items = (int)pl.items.size();
  if (n_cta) *n_cta = (int)pl.cta_begin.size();
  if (n_pages) *n_pages = (int)pl.pages.size();
  if (n_slots) *n_slots = (int)pl.csr_slots.size();
  if ((int)pl.items.size() > cap_items || (int)pl.cta_begin.size() > cap_cta ||
      (int)pl.pages.size() > cap_pages || (int)pl.csr_ptr.size() > cap_ptr ||
      (int)pl.csr_slots.size() > cap_slots)
    return fail(FK_ERR_OOM, "output capacity too small");
  if (items) std::copy(pl.items.begin(), pl.items.end(), items);
  if (cta_begin) std::copy(pl.cta_begin.begin(), pl.cta_begin.end(), cta_begin);
  if (page_ids) std::copy(pl.pages.begin(), pl.pages.end(), page_ids);
  if (csr_ptr) std::copy(pl.csr_ptr.begin(), pl.csr_ptr.end(), csr_ptr);
  if (csr_slots) std::copy(pl.csr_slots.begin(), pl.csr_slots.end(), csr_slots);
  return FK_OK;
}

fk_status fk_residual_attention(fk_pool* p, int layer, const uint16_t* q, const int32_t* agents,
                                const int32_t* bt, int max_pages, const int32_t* seq, int A,
                                int C, int causal, int compressed, uint16_t* out, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  const PoolGeom& g = p->g;
  if (layer < 0 || layer >= g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (!q || !out || !agents || !bt || !seq) return fail(FK_ERR_INVALID_ARG, "NULL argument");
  if (A < 1 || C < 1 || max_pages < 1) return fail(FK_ERR_INVALID_ARG, "A, C, max_pages must be >= 1");
  if (compressed && !g.compressed) return fail(FK_ERR_INVALID_ARG, "pool has no compressed copy");
  cudaStream_t st = (cudaStream_t)stream;
  // cache key: everything the work list depends on
  std::vector<int32_t> key;
  key.reserve(8 + 2 * A + (size_t)A * max_pages);
  key.insert(key.end(), {A, C, causal ? 1 : 0, max_pages, compressed ? 1 : 0});
  key.insert(key.end(), agents, agents + A);
  key.insert(key.end(), seq, seq + A);
  key.insert(key.end(), bt, bt + (int64_t)A * max_pages);
  if (!p->plan_valid || key != p->key) {
    p->plan_valid = false;
    std::vector<int32_t> rp(A), seen(g.max_agents, 0);
    for (int i = 0; i < A; ++i) {
      int a = agents[i];
      if (a < 0 || a >= g.max_agents || !p->agents[a].live)
        return fail(FK_ERR_INVALID_ARG, "agents[] names an unregistered agent");
      if (seen[a]++) return fail(FK_ERR_INVALID_ARG, "agents[] repeats an agent");
      if (seq[i] > p->cfg.max_tokens) return fail(FK_ERR_INVALID_ARG, "seq_len beyond rCache capacity");
      rp[i] = p->agents[a].rp;
      int np = (seq[i] + kPage - 1) / kPage;
      for (int lp = 0; lp < std::min(np, max_pages); ++lp) {
        int32_t id = bt[(int64_t)i * max_pages + lp];
        if (id >= g.num_pages || (id >= 0 && p->refcount[id] <= 0))
          return fail(FK_ERR_INVALID_ARG, "block table names a free or invalid page");
      }
    }
    HostPlan pl;
    PlanDev pd{};
    std::vector<uint8_t> blob;
    int64_t need = 0;
    fk_status s = build_call_plan(p, agents, bt, max_pages, seq, rp.data(), A, C, causal, compressed,
                                  pl, blob, pd, need);
    if (s != FK_OK) return s;
    if (need > g.ws_bytes) return fail(FK_ERR_OOM, "workspace too small for this call");
    fk_status s2 = stage_upload(p, blob.data(), blob.size(), g.base + g.off_ws, st);
    if (s2 != FK_OK) return s2;
    p->plan = std::move(pl);
    p->plan_dev = pd;
    p->key = std::move(key);
    p->plan_valid = true;
  }
  int launches = 0;
  PlanDev pd_call = p->plan_dev;
  pd_call.stall_probe = p->stall_probe ? 1 : 0;
  int e = launch_attention(g, pd_call, layer, q, out, compressed ? 1 : 0, p->num_sms,
                           stream, &launches, p->profile_event);
  if (e != 0) return cuda_fail((cudaError_t)e, "attention kernels");
  p->last_launches = launches;
  return FK_OK;
}

fk_status fk_residual_attention_noalloc(fk_pool* p, int layer, const uint16_t* q,
                                        const int32_t* agents, const int32_t* bt, int max_pages,
                                        const int32_t* seq, int A, int C, int causal,
                                        int compressed, uint16_t* out, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  const PoolGeom& g = p->g;
  if (layer < 0 || layer >= g.L) return fail(FK_ERR_INVALID_ARG, "layer out of range");
  if (!q || !out || !agents || !bt || !seq) return fail(FK_ERR_INVALID_ARG, "NULL argument");
  if (A < 1 || C < 1 || max_pages < 1) return fail(FK_ERR_INVALID_ARG, "A, C, max_pages must be >= 1");
  if (compressed && !g.compressed) return fail(FK_ERR_INVALID_ARG, "pool has no compressed copy");
  int cur_dev = -1;
  if (cudaGetDevice(&cur_dev) != cudaSuccess || cur_dev != p->device)
    return fail(FK_ERR_INVALID_ARG, "the current CUDA device is not the pool's");
  if (p->device < 0 || p->device >= kMaxDevices) return fail(FK_ERR_INVALID_ARG, "device id out of range");
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  int ce = noalloc_scratch(&scratch, &scratch_bytes);
  if (ce != 0) return cuda_fail((cudaError_t)ce, "static scratch lookup");
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<int32_t> key;
  key.reserve(8 + 2 * A + (size_t)A * max_pages);
  key.insert(key.end(), {A, C, causal ? 1 : 0, max_pages, compressed ? 1 : 0});
  key.insert(key.end(), agents, agents + A);
  key.insert(key.end(), seq, seq + A);
  key.insert(key.end(), bt, bt + (int64_t)A * max_pages);
  key.insert(key.end(), {(int32_t)(p->plan_gen & 0x7FFFFFFF), (int32_t)(p->plan_gen >> 31)});
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocCache& cache = g_noalloc[p->device];
  if (cache.pool_uid != p->uid || cache.key != key) {
    cache.pool_uid = 0;
    std::vector<int32_t> rp(A), seen(g.max_agents, 0);
    for (int i = 0; i < A; ++i) {
      int a = agents[i];
      if (a < 0 || a >= g.max_agents || !p->agents[a].live)
        return fail(FK_ERR_INVALID_ARG, "agents[] names an unregistered agent");
      if (seen[a]++) return fail(FK_ERR_INVALID_ARG, "agents[] repeats an agent");
      if (seq[i] > p->cfg.max_tokens) return fail(FK_ERR_INVALID_ARG, "seq_len beyond rCache capacity");
      rp[i] = p->agents[a].rp;
      int np = (seq[i] + kPage - 1) / kPage;
      for (int lp = 0; lp < std::min(np, max_pages); ++lp) {
        int32_t id = bt[(int64_t)i * max_pages + lp];
        if (id >= g.num_pages || (id >= 0 && p->refcount[id] <= 0))
          return fail(FK_ERR_INVALID_ARG, "block table names a free or invalid page");
      }
    }
    HostPlan pl;
    PlanDev pd{};
    std::vector<uint8_t> blob;
    int64_t need = 0;
    fk_status s = build_call_plan(p, agents, bt, max_pages, seq, rp.data(), A, C, causal, compressed,
                                  pl, blob, pd, need);
    if (s != FK_OK) return s;
    if (need > (int64_t)scratch_bytes) {
      char msg[160];
      std::snprintf(msg, sizeof msg,
                    "call needs %lld bytes of scratch; the static array holds %zu",
                    (long long)need, scratch_bytes);
      return fail(FK_ERR_OOM, msg);
    }
    // pageable source, kept in the cache entry until the next upload
    cache.blob = std::move(blob);
    cudaError_t e = cudaMemcpyAsync(scratch, cache.blob.data(), cache.blob.size(),
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "work list upload");
    cache.pool_uid = p->uid;
    cache.key = std::move(key);
    cache.pd = pd;
  }
  PoolGeom g2 = g;
  g2.off_ws = (int64_t)((uint8_t*)scratch - g.base);
  g2.ws_bytes = (int64_t)scratch_bytes;
  int launches = 0;
  PlanDev pd_call = cache.pd;
  pd_call.stall_probe = p->stall_probe ? 1 : 0;
  int e = launch_attention(g2, pd_call, layer, q, out, compressed ? 1 : 0, p->num_sms, stream,
                           &launches, nullptr);
  if (e != 0) return cuda_fail((cudaError_t)e, "attention kernels");
  p->last_launches = launches;
  return FK_OK;
}

int fk_last_launch_count(const fk_pool* p) { return p ? p->last_launches : 0; }

fk_status fk_pool_set_test_stall(fk_pool* p, int on) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  p->stall_probe = on != 0;
  return FK_OK;
}

fk_status fk_pool_set_profile_event(fk_pool* p, void* event) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  p->profile_event = event;
  return FK_OK;
}

fk_status fk_check(fk_pool* p, void* stream) {
  if (!p) return fail(FK_ERR_INVALID_ARG, "pool is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word[3] = {0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(word, p->g.base + p->g.off_err, 12, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "fk_check");
  if (word[0] || word[1]) {
    cudaMemsetAsync(p->g.base + p->g.off_err, 0, 12, st);
    cudaStreamSynchronize(st);
    char msg[160];
    std::snprintf(msg, sizeof msg,
                  "device check fired: bounds 0x%x, waits %u (first: warp %u, barrier smem 0x%x)",
                  word[0], word[1], (word[2] >> 20) & 0x7FFu, word[2] & 0xFFFFFu);
    return fail(word[1] ? FK_ERR_TIMEOUT : FK_ERR_DEVICE_CHECK, msg);
  }
  return FK_OK;
}

}  // extern "C"
