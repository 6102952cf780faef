// Residual attention for calls with many query rows per agent and kv head
// (a causal chunk of C tokens times the G query heads of a kv head, e.g.
// 32 x 8 = 256 rows): the work is a dense contraction, so each work item
// takes 128 rows of one agent (the MMA's M) and walks its keys in
// 128-token tiles.
//
// ForkKV guide, "Mathematical Formulation of ResidualAttention" and "On-the-
// Fly Register Fusion": the adapted key is the shared base key plus the
// rotated low-rank residual, K_a[t] = Kb[t] + s RoPE_t(Lk[t] Bk); the value
// residual stays factored (LRAgent summary, section 3): O = P Vb and
// OL = P Lv are accumulated separately and Bv is applied once per row by
// the combine kernel.
//
// Per 128-key tile:
//   warp 0       bulk-copies the tile's Lk rows, Kb pages and then Vb pages
//                and Lv rows (one 4 KB block per page, one block of rows);
//   warp 1       S = Q K_a^T (rows x keys); U = Lk BkT of the next tile
//                (keys x d, fp32); O += P Vb and OL += P Lv of the previous
//                tile, with P read from TMEM;
//   warp 2       the rotation of each tile's first key, cos and sin of
//                t0 theta_i reduced exactly through a 64-bit fraction of a
//                turn, one tile ahead;
//   warps 4-7,   one thread per key and half of the frequencies (warps
//   12-15        4-7 the first 32, warps 12-15 the last 32): K_a = Kb +
//                s RoPE_t(U) rounded to bf16, written over the tile's Kb in
//                shared memory; the key's rotation is the tile's composed
//                with the key's own offset rotation (kept in registers for
//                the whole kernel);
//   warps 8-11   one thread per row: masked online softmax of S (base 2;
//                O and OL are rescaled in TMEM only when a row's running
//                maximum grows by more than 2^8), P in bf16 into TMEM; at
//                the end of an item, the row's split partial (m, l, O, OL).
// Every wait is bounded: a timeout sets the pool's error word and the CTA
// abort flag, and the CTA leaves after a grace period for copies in flight.
#include <cuda_runtime.h>

#include <cstdint>

#include "fk_device.cuh"
#include "fk_internal.h"
#include "fk_once.h"

namespace fk {
namespace chk {

constexpr int D = 128;
constexpr int kThreads = 512;
constexpr int kRMax = 64;                       // padded rank limit
constexpr uint32_t kTmU = 0, kTmS = 128, kTmO = 256, kTmOL = 384, kTmP = 448;

struct Layout {
  static constexpr int PAGE_B = kPage * D * 2;            // one (page, head) block: 4 KB
  static constexpr int KB_B = kTilePages * PAGE_B;        // a tile's keys, rewritten in place as K_a
  static constexpr int VB_B = KB_B;
  static constexpr int LR_B = kTileTok * kRMax * 2;       // a tile's Lk or Lv rows
  static constexpr int Q_B = 128 * D * 2;
  static constexpr int BK_B = D * kRMax * 2;
  static constexpr int oKB0 = 0;
  static constexpr int oKB1 = oKB0 + KB_B;
  static constexpr int oVB0 = oKB1 + KB_B;
  static constexpr int oVB1 = oVB0 + VB_B;
  static constexpr int oLV0 = oVB1 + VB_B;
  static constexpr int oLV1 = oLV0 + LR_B;
  static constexpr int oLK = oLV1 + LR_B;
  static constexpr int oQ = oLK + LR_B;
  static constexpr int oBK = oQ + Q_B;
  static constexpr int oMISC = oBK + BK_B;
  static constexpr int MISC_B = 2048;
  static constexpr int TOTAL = oMISC + MISC_B;
};
static_assert(Layout::TOTAL <= 232448, "shared memory over the 227 KB a CTA may use");

enum {
  B_KB_FULL0, B_KB_FULL1, B_KB_EMPTY0, B_KB_EMPTY1, B_LK_FULL, B_LK_EMPTY, B_V_FULL0, B_V_FULL1,
  B_V_EMPTY0, B_V_EMPTY1, B_BK_FULL, B_BK_EMPTY, B_Q_FULL, B_U_FULL, B_U_FREE, B_KA_READY,
  B_S_FULL, B_S_FREE, B_P_FULL, B_PV_DONE, B_ACC_EMPTY, B_FINAL, B_ROT_FULL0, B_ROT_FULL1,
  B_ROT_EMPTY0, B_ROT_EMPTY1, B_COUNT
};
// arrivals: one lane per warp of one or two warpgroups, else one thread or
// a commit
__host__ __device__ constexpr uint32_t bar_count(int i) {
  return (i == B_U_FREE || i == B_KA_READY || i == B_ROT_EMPTY0 || i == B_ROT_EMPTY1)
             ? 8u   // both key warpgroups
             : (i == B_Q_FULL || i == B_S_FREE || i == B_P_FULL || i == B_ACC_EMPTY) ? 4u : 1u;
}
// barriers a role waits on as "empty" start one phase ahead
constexpr uint32_t kEmptyMask = (1u << B_KB_EMPTY0) | (1u << B_KB_EMPTY1) | (1u << B_LK_EMPTY) |
                                (1u << B_V_EMPTY0) | (1u << B_V_EMPTY1) | (1u << B_BK_EMPTY) |
                                (1u << B_U_FREE) | (1u << B_S_FREE) | (1u << B_ACC_EMPTY) |
                                (1u << B_ROT_EMPTY0) | (1u << B_ROT_EMPTY1);

struct Misc {
  uint64_t bar[B_COUNT];
  unsigned long long frac[64];   // theta_i / (2 pi) as a 64-bit binary fraction
  float2 rot[2][64];             // (cos, sin) of t0 theta_i, a ring of two tiles
  float theta[64];               // theta_i
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Misc) <= Layout::MISC_B, "Misc must fit its smem slot");

// the two bf16 halves of a 32-bit word as fp32 (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// What every role derives from a work item of the chunk plan: one call
// agent, one kv head, rows row_begin .. row_begin + n_rows - 1 of that
// agent's G*C rows (row index c*G + g), logical pages lp_begin ..
struct Item {
  int head, row_begin, n_rows, page_begin, n_pages, lp_begin, agent, partial_begin, n_tiles;
  int pool_agent, T, rp;
  float s;
  int64_t rc_off;
};

__device__ __forceinline__ void load_item(const PoolGeom& g, const PlanDev& p, const uint8_t* ws,
                                          int it, Item& I) {
  const fk_work_item& w = ((const fk_work_item*)(ws + p.off_items))[it];
  const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
  const AgentDev* ag = (const AgentDev*)(g.base + g.off_agents);
  I.head = w.head;
  I.row_begin = w.row_begin;
  I.n_rows = w.n_rows;
  I.page_begin = w.page_begin;
  I.n_pages = w.n_pages;
  I.lp_begin = w.lp_begin;
  I.agent = w.agent_begin;
  I.partial_begin = w.partial_begin;
  I.n_tiles = (w.n_pages + kTilePages - 1) / kTilePages;
  const CallAgent c = ca[I.agent];
  I.pool_agent = c.pool_agent;
  I.T = c.seq_len;
  const AgentDev dv = ag[c.pool_agent];
  I.rp = dv.rp;
  I.s = dv.s;
  I.rc_off = dv.rc_off;
}

}  // namespace chk

__global__ void __launch_bounds__(chk::kThreads, 1)
    chunk_kernel(PoolGeom g, PlanDev p, int layer, const uint16_t* __restrict__ q) {
  using namespace chk;
  using LY = Layout;
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc& M = *(Misc*)(smem + LY::oMISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* ws = g.base + g.off_ws;
  const int32_t* cta_items = (const int32_t*)(ws + p.off_cta);
  uint32_t* errw = (uint32_t*)(g.base + g.off_err);
  volatile int* abort_flag = &M.abort_flag;
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&M.bar[i]); };
  uint32_t ph = kEmptyMask;   // bit i: the parity this role waits for next on barrier i
  auto wait = [&](int i) {
    uint32_t par = (ph >> i) & 1u;
    const bool ok = mbar_wait(bar(i), par, abort_flag, errw);
    ph ^= 1u << i;
    return ok;
  };
  // the dependent combine grid may be scheduled now; it waits for this
  // grid's completion before reading the partials
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- set-up: zero smem (stale rows read by masked keys stay finite),
  // RoPE fractions, barriers, TMEM
  for (int i = tid * 16; i < LY::oMISC; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  if (tid < 64) {
    M.theta[tid] = ((const float*)(g.base + g.off_rope))[tid];
    M.frac[tid] = ((const unsigned long long*)(g.base + g.off_rope + 256))[tid];
  }
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), bar_count(i));
    M.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&M.tmem_base), 512);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_base;
  const int it_begin = cta_items[blockIdx.x], it_end = cta_items[blockIdx.x + 1];

  if (warp == 0) {
    // ============================================================ loads ====
    if (lane == 0) {
      int tc = 0;
      for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
        Item I;
        load_item(g, p, ws, it, I);
        const int32_t* pages = (const int32_t*)(ws + p.off_pages) + I.page_begin;
        const uint8_t* lk = g.base + I.rc_off + (int64_t)layer * rc_layer_bytes(g, I.rp);
        const uint8_t* lv = lk + (int64_t)g.tcap * I.rp * 2;
        if (!wait(B_BK_EMPTY)) break;
        mbar_expect_tx(bar(B_BK_FULL), D * I.rp * 2);
        bulk_g2s(sbase + LY::oBK,
                 g.base + g.off_bk + (int64_t)I.pool_agent * g.bk_agent_bytes +
                     ((int64_t)layer * g.H_kv + I.head) * (int64_t)D * g.rmax_pad * 2,
                 D * I.rp * 2, bar(B_BK_FULL));
        bool ok = true;
        for (int k = 0; k < I.n_tiles && ok; ++k, ++tc) {
          const int kb = tc & 1;
          const int p0 = k * kTilePages;
          const int np = min(kTilePages, I.n_pages - p0);
          const int t0 = (I.lp_begin + p0) * kPage;
          const int nr = min(kTileTok, g.tcap - t0);          // rCache rows of the tile
          // Lk (freed by the previous tile's U), Kb (freed by the S of two
          // tiles back), Vb and Lv (freed by the PV of two tiles back)
          if (!wait(B_LK_EMPTY)) { ok = false; break; }
          mbar_expect_tx(bar(B_LK_FULL), nr * I.rp * 2);
          bulk_g2s(sbase + LY::oLK, lk + (int64_t)t0 * I.rp * 2, nr * I.rp * 2, bar(B_LK_FULL));
          if (!wait(B_KB_EMPTY0 + kb)) { ok = false; break; }
          mbar_expect_tx(bar(B_KB_FULL0 + kb), np * LY::PAGE_B);
          for (int j = 0; j < np; ++j)
            bulk_g2s(sbase + (kb ? LY::oKB1 : LY::oKB0) + j * LY::PAGE_B,
                     g.base + g.off_kb + (int64_t)layer * g.kb_layer_bytes +
                         ((int64_t)pages[p0 + j] * g.H_kv + I.head) * LY::PAGE_B,
                     LY::PAGE_B, bar(B_KB_FULL0 + kb));
          if (!wait(B_V_EMPTY0 + kb)) { ok = false; break; }
          mbar_expect_tx(bar(B_V_FULL0 + kb), np * LY::PAGE_B + nr * I.rp * 2);
          for (int j = 0; j < np; ++j)
            bulk_g2s(sbase + (kb ? LY::oVB1 : LY::oVB0) + j * LY::PAGE_B,
                     g.base + g.off_vb + (int64_t)layer * g.kb_layer_bytes +
                         ((int64_t)pages[p0 + j] * g.H_kv + I.head) * LY::PAGE_B,
                     LY::PAGE_B, bar(B_V_FULL0 + kb));
          bulk_g2s(sbase + (kb ? LY::oLV1 : LY::oLV0), lv + (int64_t)t0 * I.rp * 2, nr * I.rp * 2,
                   bar(B_V_FULL0 + kb));
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================================================= MMAs ====
    if (lane == 0) {
      int tc = 0;
      const uint32_t t_U = tmem + kTmU, t_S = tmem + kTmS, t_O = tmem + kTmO, t_OL = tmem + kTmOL;
      const uint32_t idK = idesc_f16(128, 128, 1);
      for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
        Item I;
        load_item(g, p, ws, it, I);
        const uint32_t idL = idesc_f16(128, I.rp, 1);
        if (!wait(B_BK_FULL) || !wait(B_Q_FULL)) break;
        tc_fence_after();
        // U = Lk BkT of tile k: keys x d, K = padded rank
        auto issue_u = [&](int k) {
          if (!wait(B_LK_FULL) || !wait(B_U_FREE)) return false;
          tc_fence_after();
          for (int ks = 0; ks < I.rp / 16; ++ks)
            mma_ss(t_U, sdesc(sbase + LY::oLK + ks * 256, 128, I.rp * 16),
                   sdesc(sbase + LY::oBK + ks * 256, 128, I.rp * 16), idK, ks > 0 ? 1u : 0u);
          mma_commit(bar(B_U_FULL));
          mma_commit(bar(B_LK_EMPTY));
          if (k == I.n_tiles - 1) mma_commit(bar(B_BK_EMPTY));
          return true;
        };
        // O += P Vb, OL += P Lv of tile j (P from TMEM, bf16 pairs)
        auto issue_pv = [&](int j) {
          const int kb = (tc + j) & 1;
          if (!wait(B_P_FULL) || !wait(B_V_FULL0 + kb)) return false;
          if (j == 0 && !wait(B_ACC_EMPTY)) return false;
          tc_fence_after();
          const uint32_t vbase = sbase + (kb ? LY::oVB1 : LY::oVB0);
          const uint32_t lvbase = sbase + (kb ? LY::oLV1 : LY::oLV0);
#pragma unroll
          for (int ks = 0; ks < kTileTok / 16; ++ks) {
            const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
            mma_ts(t_O, tmem + kTmP + 8 * ks, sdesc(vbase + ks * 2 * (D / 8) * 128, (D / 8) * 128, 128),
                   idK, acc);
            mma_ts(t_OL, tmem + kTmP + 8 * ks, sdesc(lvbase + ks * 2 * I.rp * 16, I.rp * 16, 128), idL,
                   acc);
          }
          mma_commit(bar(B_PV_DONE));
          mma_commit(bar(B_V_EMPTY0 + kb));
          return true;
        };
        bool ok = issue_u(0);
        for (int k = 0; k < I.n_tiles && ok; ++k) {
          const int kb = (tc + k) & 1;
          // S = Q K_a^T: rows x keys, K = d; the stage's keys are free after it
          if (!wait(B_KA_READY) || !wait(B_S_FREE)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kbase = sbase + (kb ? LY::oKB1 : LY::oKB0);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss(t_S, sdesc(sbase + LY::oQ + ks * 256, 128, (D / 8) * 128),
                   sdesc(kbase + ks * 256, 128, (D / 8) * 128), idK, ks > 0 ? 1u : 0u);
          mma_commit(bar(B_S_FULL));
          mma_commit(bar(B_KB_EMPTY0 + kb));
          if (k + 1 < I.n_tiles && !issue_u(k + 1)) { ok = false; break; }
          if (k >= 1 && !issue_pv(k - 1)) { ok = false; break; }
        }
        if (ok) ok = issue_pv(I.n_tiles - 1);
        tc += I.n_tiles;
        if (!ok) break;
      }
      // every MMA issued has completed before TMEM is released
      mma_commit(bar(B_FINAL));
      uint32_t par = (ph >> B_FINAL) & 1u;
      if (!mbar_wait_drain(bar(B_FINAL), par)) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 2) {
    // ============================== tile-start rotations, one tile ahead ====
    int tc = 0;
    for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
      Item I;
      load_item(g, p, ws, it, I);
      bool ok = true;
      for (int k = 0; k < I.n_tiles; ++k, ++tc) {
        const int b = tc & 1;
        if (!__all_sync(0xffffffffu, wait(B_ROT_EMPTY0 + b))) { ok = false; break; }
        const unsigned long long t0 = (unsigned long long)((I.lp_begin + k * kTilePages) * kPage);
#pragma unroll
        for (int z = 0; z < 2; ++z) {
          const int i = 2 * lane + z;
          const unsigned long long fr = t0 * M.frac[i];
          float ang = (float)(unsigned int)(fr >> 32) * 1.4629180792671596e-09f;   // 2 pi / 2^32
          if (ang > 3.14159265f) ang -= 6.28318531f;
          float sn, cs;
          sincosf(ang, &sn, &cs);
          M.rot[b][i] = make_float2(cs, sn);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ROT_FULL0 + b));
      }
      if (!ok) break;
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // =============================================== adapted keys K_a ====
    const int kl = 32 * (warp & 3) + lane;                 // TMEM lane = key of the tile
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int f0 = warp >= 12 ? 32 : 0;                    // this warpgroup's first frequency
    // the rotation by this key's offset in its tile, (cos, sin) of kl theta_i
    // as f16 pairs, for the whole kernel
    uint32_t tau[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float sn, cs;
      sincosf((float)kl * M.theta[f0 + i], &sn, &cs);
      tau[i] = pack_h2(cs, sn);
    }
    int tc = 0;
    for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
      Item I;
      load_item(g, p, ws, it, I);
      bool ok = true;
      for (int k = 0; k < I.n_tiles; ++k, ++tc) {
        const int kb = tc & 1, b = tc & 1;
        // (lanes leave together: the TMEM accesses below are warp-wide)
        if (!__all_sync(0xffffffffu, wait(B_ROT_FULL0 + b) & wait(B_KB_FULL0 + kb) & wait(B_U_FULL))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* krow = smem + (kb ? LY::oKB1 : LY::oKB0) + (kl / 8) * ((D / 8) * 128) + (kl % 8) * 16;
#pragma unroll
        for (int jq = 0; jq < 4; ++jq) {
          // frequencies f0 + 8 jq .. + 7: d columns i (chunk jg) and i + 64 (chunk 8 + jg)
          const int jg = f0 / 8 + jq;
          uint32_t ulo[8], uhi[8];
          tmem_ld8(tmem + kTmU + 8 * jg + lane_off, ulo);
          tmem_ld8(tmem + kTmU + 64 + 8 * jg + lane_off, uhi);
          tmem_wait_ld();
          if (jq == 3) {
            // U read: the next tile's U may be written
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_U_FREE));
          }
          const uint4 klo = *(const uint4*)(krow + jg * 128);
          const uint4 khi = *(const uint4*)(krow + (8 + jg) * 128);
          uint32_t lo_w[4] = {klo.x, klo.y, klo.z, klo.w};
          uint32_t hi_w[4] = {khi.x, khi.y, khi.z, khi.w};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float klf[2], khf[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e2 + h, i = 8 * jq + e;
              // rotation of key t0 + kl: the tile start's composed with the offset's
              const float2 r0 = M.rot[b][f0 + i];
              const float2 rt = __half22float2(*reinterpret_cast<const __half2*>(&tau[i]));
              const float cs = r0.x * rt.x - r0.y * rt.y;
              const float sn = r0.y * rt.x + r0.x * rt.y;
              const float ul = __uint_as_float(ulo[e]), uh = __uint_as_float(uhi[e]);
              const float bl = h ? bf_hi(lo_w[e2]) : bf_lo(lo_w[e2]);
              const float bh = h ? bf_hi(hi_w[e2]) : bf_lo(hi_w[e2]);
              klf[h] = bl + I.s * (ul * cs - uh * sn);
              khf[h] = bh + I.s * (uh * cs + ul * sn);
            }
            lo_w[e2] = pack_bf2(klf[0], klf[1]);
            hi_w[e2] = pack_bf2(khf[0], khf[1]);
          }
          *(uint4*)(krow + jg * 128) = make_uint4(lo_w[0], lo_w[1], lo_w[2], lo_w[3]);
          *(uint4*)(krow + (8 + jg) * 128) = make_uint4(hi_w[0], hi_w[1], hi_w[2], hi_w[3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_ROT_EMPTY0 + b));
          mbar_arrive(bar(B_KA_READY));
        }
      }
      if (!ok) break;
    }
  } else if (warp >= 8) {
    // ====================================================== softmax ====
    const int r = tid - 256;                               // TMEM lane = query row
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)D);
    float* part = (float*)(ws + p.off_partials);
    const int PS = p.partial_stride;
    auto ex2 = [](float x) {
      float y;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
      return y;
    };
    int tc = 0;
    for (int it = it_begin; it < it_end && !*abort_flag; ++it) {
      Item I;
      load_item(g, p, ws, it, I);
      const bool valid = r < I.n_rows;
      const int ridx = I.row_begin + r;
      const int c = ridx / g.G, gq = ridx % g.G;
      const int pos = p.causal ? I.T - p.C + c : 0x7fffffff;
      const int lim = min(I.T, pos == 0x7fffffff ? I.T : pos + 1);   // keys t < lim are visible
      // ---- Q rows (the previous item's S MMAs have completed: their S_FULL was seen)
      {
        const int64_t qrow = ((int64_t)I.agent * p.C + c) * g.H_q + I.head * g.G + gq;
#pragma unroll 4
        for (int ch = 0; ch < D / 8; ++ch) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (valid) v = *(const uint4*)(q + qrow * D + ch * 8);
          *(uint4*)(smem + LY::oQ + ((r / 8) * (D / 8) + ch) * 128 + (r % 8) * 16) = v;
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_Q_FULL));
      }
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      for (int k = 0; k < I.n_tiles; ++k, ++tc) {
        const int t0 = (I.lp_begin + k * kTilePages) * kPage;
        const int ntok = min(kTileTok, (I.n_pages - k * kTilePages) * kPage);
        const int nvis = valid ? max(0, min(ntok, lim - t0)) : 0;   // keys 0 .. nvis-1 count
        if (!__all_sync(0xffffffffu, wait(B_S_FULL))) { ok = false; break; }
        tc_fence_after();
        // pass 1: the tile's row maximum (two loads in flight; the scale is
        // positive, so it is applied to the maximum only)
        const bool full = nvis == kTileTok;                // no key of the tile is masked
        float tmax = -INFINITY;
#pragma unroll 1
        for (int cb = 0; cb < kTileTok; cb += 64) {
          uint32_t v[64];
          tmem_ld32(tmem + kTmS + cb + lane_off, v);
          tmem_ld32(tmem + kTmS + cb + 32 + lane_off, v + 32);
          tmem_wait_ld();
          if (full) {
#pragma unroll
            for (int e = 0; e < 64; ++e) tmax = fmaxf(tmax, __uint_as_float(v[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (cb + e < nvis) tmax = fmaxf(tmax, __uint_as_float(v[e]));
          }
        }
        if (tmax != -INFINITY) tmax *= scale_log2;
        bool rescale = false;
        float alpha = 1.f;
        if (m_used == -INFINITY) {
          m_used = tmax;
        } else if (tmax > m_used + 8.f) {
          alpha = ex2(m_used - tmax);
          m_used = tmax;
          rescale = true;
        }
        // every accumulation is waited for in order (the previous tile's,
        // here): then O, OL shrink by alpha if the maximum moved, and this
        // tile's P replaces the previous one in TMEM
        if (k > 0) {
          if (!__all_sync(0xffffffffu, wait(B_PV_DONE))) { ok = false; break; }
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {    // warp-wide; alpha is 1 in the other lanes
#pragma unroll 1
            for (int cb = 0; cb < D + kRMax; cb += 32) {
              if (cb >= D && cb - D >= I.rp) break;
              const uint32_t col = cb < D ? kTmO + cb : kTmOL + (cb - D);
              uint32_t v[32];
              tmem_ld32_wait(tmem + col + lane_off, v);
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(tmem + col + lane_off, v);
            }
          }
        }
        // pass 2: P = 2^(s - m) as bf16 pairs into TMEM (key 2j, 2j + 1 in
        // column j), and the row sum (fp32, before the rounding to bf16)
        float lt = 0.f;
        const float nm = m_used == -INFINITY ? 0.f : -m_used;
#pragma unroll 1
        for (int cb = 0; cb < kTileTok; cb += 32) {
          uint32_t v[32], w[16];
          tmem_ld32_wait(tmem + kTmS + cb + lane_off, v);
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = ex2(fmaf(__uint_as_float(v[e]), scale_log2, nm));
              const float p1 = ex2(fmaf(__uint_as_float(v[e + 1]), scale_log2, nm));
              w[e / 2] = pack_bf2(p0, p1);
              lt += p0 + p1;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float p0 = (cb + e < nvis) ? ex2(fmaf(__uint_as_float(v[e]), scale_log2, nm)) : 0.f;
              const float p1 = (cb + e + 1 < nvis) ? ex2(fmaf(__uint_as_float(v[e + 1]), scale_log2, nm)) : 0.f;
              w[e / 2] = pack_bf2(p0, p1);
              lt += p0 + p1;
            }
          }
          tmem_st16(tmem + kTmP + cb / 2 + lane_off, w);
        }
        tmem_wait_st();
        l = l * alpha + lt;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_S_FREE));
          mbar_arrive(bar(B_P_FULL));
        }
      }
      if (!ok) break;
      // ---- the item's split partials, once its last accumulation completed
      {
        if (!__all_sync(0xffffffffu, wait(B_PV_DONE))) break;
        tc_fence_after();
        float* dst = part + (int64_t)(I.partial_begin + r) * PS;
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t v[32];
          tmem_ld32_wait(tmem + kTmO + cb + lane_off, v);
          if (valid)
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[4 + cb + e] = __uint_as_float(v[e]);
        }
#pragma unroll 1
        for (int cb = 0; cb < I.rp; cb += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + kTmOL + cb + lane_off, v);
          tmem_wait_ld();
          if (valid)
#pragma unroll
            for (int e = 0; e < 16; ++e) dst[4 + D + cb + e] = __uint_as_float(v[e]);
        }
        if (valid) {
          dst[0] = m_used;
          dst[1] = l;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY));
      }
    }
  }
  // ---- tear-down.  After a timed-out wait, give bulk copies still in
  // flight a bounded grace period before the CTA's smem is released.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) { }
  }
  if (warp == 1) tmem_dealloc(tmem, 512);
}

bool chunk_applies(const PoolGeom& g, const PlanDev& p) { return p.chunk != 0 && g.d == chk::D; }

int launch_chunk(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q, void* stream) {
  static PerDeviceOnce once;
  const int se = once.run([] {
    return (int)cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     chk::Layout::TOTAL);
  });
  if (se != 0) return se;
  chunk_kernel<<<p.n_ctas, chk::kThreads, chk::Layout::TOTAL, (cudaStream_t)stream>>>(g, p, layer, q);
  return (int)cudaGetLastError();
}

}  // namespace fk
