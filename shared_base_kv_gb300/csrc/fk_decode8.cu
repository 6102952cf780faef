// Residual attention for decode-shaped calls over tiles of up to eight
// agents (four query rows per agent and kv head, d = 128): every (page, kv
// head) block of the shared base cache is streamed from HBM once and scored
// against all 32 query rows of the tile.
//
// Scores (ForkKV guide, "Mathematical Formulation of ResidualAttention"):
//     q . (Kb[t] + s RoPE_t(Lk[t] Bk)) / sqrt(d).
// The base part S = Kb Q^T is one tensor-core contraction per 128-key tile
// (N = 32 rows).  RoPE is linear and acts per frequency pair (i, i + d/2),
// so the residual part regroups on the query side:
//     q . RoPE_t(Lk[t] Bk) = sum_k Lk[t,k] Z[t,(k,g)],   Z = Trig(t) M,
// Trig(t) = [cos t th_i, sin t th_i] (128 keys x d) and M (d x 4 sum-of-ranks)
// built from s q and Bk once per work item.  Z runs on the tensor cores with
// Trig read from tensor memory; the length-r sums against Lk run on the CUDA
// cores next to the softmax.  With all agents of a tile in one pass, the
// shared contractions (S, P Vb) use N = 32 and every base page is read once.
//
// Values keep the factored form (LRAgent summary, section 3): O^T = Vb^T P
// and OL^T = Lv^T P on the tensor cores (Lv^T held in tensor memory), Bv
// applied once per row in the combine.  Row sums of P are warp reductions.
//
// Warp roles (512 threads):
//   warp 0       bulk copies of key pages (one stage); L2 prefetch of the
//                item's Lk and Lv rows a tile ahead
//   warp 3       bulk copies of value pages (one stage)
//   warp 1       MMA issue (converged warp, elect.sync)
//   warps 4-7    compute warpgroup 0: agent slots 0-3 (rows 0-15)
//   warps 8-11   compute warpgroup 1: agent slots 4-7 (rows 16-31)
//   warps 12-15  Trig warpgroup: Trig of each tile (from the pool's table of
//                per-position rotations) and the tile's Lv^T into tensor
//                memory
// The compute and Trig warpgroups build M in shared memory at the start of
// every work item.  A warp reaches TMEM lanes 32 (warp % 4) .. + 31, so the
// thread of TMEM lane 32 (warp % 4) + lane handles the key (or d, or rank
// slot) of that lane.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fk_device.cuh"
#include "fk_internal.h"
#include "fk_once.h"

namespace fk {
namespace d8 {

constexpr int D = 128;
constexpr int NF = D / 2;                   // RoPE frequencies
constexpr int kThreads = 512;
constexpr int kSlots = kDecodeSlots;        // agent slots of a tile
constexpr int kRPA = 4;                     // query rows per agent slot
constexpr int kRows = kSlots * kRPA;        // 32
constexpr int kWGGroups = 8;                // 8-rank groups of one compute warpgroup (64 ranks)
constexpr int kMaxGroups = 2 * kWGGroups;   // 8-rank groups of a tile (128 ranks)
constexpr int kMaxZ = kRPA * 8 * kMaxGroups;   // 512 Z columns: (rank, row) pairs

// TMEM columns: base scores S (32 rows), O^T (d lanes x 32 rows), OL^T
// (rank lanes x 32 rows), Lv^T (rank lanes x 128 keys as bf16 pairs), Trig
// (key lanes x 64 f16 pairs), and one Z buffer of 128 columns per compute
// warpgroup (a chunk of four 8-rank groups).  A tensor-core accumulator
// that changes from one MMA run to the next costs time (measured on GB300:
// N = 64 MMAs of eight-deep runs into rotating buffers ran at 61 cycles
// each against 35 into one buffer), so Z runs in as few, as wide chunks as
// tensor memory holds.
constexpr uint32_t kTmS = 0, kTmO = 32, kTmOL = 64, kTmLv = 96, kTmTrig = 160, kTmZ = 224;
constexpr int kZChunkGroups = 4;
constexpr uint32_t kZBufCols = 32 * kZChunkGroups;
__host__ __device__ constexpr uint32_t tm_z(int wg) { return kTmZ + kZBufCols * (uint32_t)wg; }
static_assert(kTmZ + 2 * kZBufCols <= 512, "TMEM map");

// Shared memory.  M: K-major core matrices of 8 Z columns x 8 features
// (f16, features 2i / 2i + 1 the cos / sin parts of frequency i).  Kb and
// Vb: one 128-key stage each, pages in the pool's tensor-core layouts.  Q:
// bf16 rows, the B operand of S.  P: two buffers of bf16 P (row groups of
// 16 key chunks, 144-byte core matrices against bank conflicts).
constexpr int PAGE_B = kPage * D * 2;
constexpr int TILE_B = kTilePages * PAGE_B;
constexpr int M_B = kMaxZ * D * 2;
constexpr int kPChunk = 144;
constexpr int kPRowGroup = 16 * kPChunk;
constexpr int P_B = (kRows / 8) * kPRowGroup;
constexpr int Q_B = kRows * D * 2;
constexpr int oM = 0;
constexpr int oKB = oM + M_B;
constexpr int oVB = oKB + TILE_B;
constexpr int oQ = oVB + TILE_B;
constexpr int oP = oQ + Q_B;
constexpr int oMISC = oP + 2 * P_B;
constexpr int MISC_B = 6144;
constexpr int TOTAL = oMISC + MISC_B;
static_assert(oMISC % 128 == 0, "misc block alignment");
static_assert(TOTAL <= 232448, "shared memory over the 227 KB a CTA may use");

enum {
  B_KB_FULL, B_KB_EMPTY, B_VB_FULL, B_VB_EMPTY, B_LV_FULL, B_LV_EMPTY, B_Q_FULL, B_M_FULL,
  B_TRIG_FULL, B_TRIG_EMPTY, B_S_FULL, B_S_FREE, B_ZF0, B_ZF1, B_ZE0, B_ZE1,
  B_P_FULL0, B_P_FULL1, B_PV_DONE0, B_PV_DONE1, B_ACC_EMPTY, B_FINAL, B_COUNT
};
// Z buffer of compute warpgroup w: full (MMA commit) and free (the
// warpgroup's four warps).
__host__ __device__ constexpr int b_zf(int w) { return B_ZF0 + w; }
__host__ __device__ constexpr int b_ze(int w) { return B_ZE0 + w; }
// Arrival counts: 8 = lane 0 of each compute warp; 12 = compute and Trig
// warps; 4 = lane 0 of each warp of one warpgroup; 1 = a transaction count
// or an MMA commit.
__host__ __device__ constexpr uint32_t bar_count(int i) {
  return (i == B_S_FREE || i == B_P_FULL0 || i == B_P_FULL1 || i == B_ACC_EMPTY || i == B_Q_FULL)
             ? 8u
         : (i == B_M_FULL) ? 12u
         : (i == B_TRIG_FULL || i == B_LV_FULL || i == B_ZE0 || i == B_ZE1) ? 4u
                                                                               : 1u;
}
// Barriers whose first wait must pass at once (a free buffer).
constexpr uint64_t kEmptyMask = (1ull << B_KB_EMPTY) | (1ull << B_VB_EMPTY) |
                                (1ull << B_LV_EMPTY) | (1ull << B_ZE0) | (1ull << B_ZE1) |
                                (1ull << B_S_FREE) | (1ull << B_ACC_EMPTY);
static_assert(B_COUNT <= 64, "one parity bit per barrier");

struct Misc {
  uint64_t bar[B_COUNT];
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float m_used[kRows];   // (16-byte aligned: read as float4)
  float alpha[kRows];
  float red[4][kRows];               // per warp of a warpgroup: row maxima, row sums
  alignas(16) int32_t row_lim[kRows];  // key t is visible to row j iff t < row_lim[j]
  int32_t lim_min[2];                // smallest row_lim of each warpgroup (0: a padded row)
  int32_t mslot[kMaxGroups];         // slot owning 8-rank group j of the tile
  int32_t half_groups[2];            // 8-rank groups of each compute warpgroup's slots
  // the item's slots (written by compute warpgroup 0 at the item's start):
  // padded rank (0: empty slot), first rank column, pool agent, scale,
  // rCache offset
  int32_t srp[kSlots], scol[kSlots], spa[kSlots];
  float ss[kSlots];
  int64_t src[kSlots];
  // per compute warpgroup and local 8-rank group: address of key t's 8
  // ranks is gbase + (t / 8) * gstride + (t % 8) * 16; gslot = slot - 4 cw
  const uint8_t* gbase[2][kWGGroups];
  int32_t gstride[2][kWGGroups];
  int32_t gslot[2][kWGGroups];
};
static_assert(sizeof(Misc) <= MISC_B, "Misc must fit its smem slot");
static_assert(offsetof(Misc, m_used) % 16 == 0 && offsetof(Misc, row_lim) % 16 == 0,
              "tables read as 16-byte vectors");

// One work item: a tile of agent slots (rank 0: empty), a kv head and a run
// of the tile's shared pages.
struct Item {
  int head, n_pages, lp_begin, page_begin, n_tiles, partial_begin, row_begin, sum_rp, n_groups;
  int rp[kSlots], col[kSlots], pa[kSlots];
  float s[kSlots];
  int64_t rc_off[kSlots];
};

__device__ __forceinline__ void load_item(const PoolGeom& g, const PlanDev& p, const uint8_t* ws,
                                          int it, Item& I) {
  const fk_work_item& w = ((const fk_work_item*)(ws + p.off_items))[it];
  const int32_t* tile_agents = (const int32_t*)(ws + p.off_tile_agents);
  const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
  const AgentDev* ag = (const AgentDev*)(g.base + g.off_agents);
  I.head = w.head;
  I.n_pages = w.n_pages;
  I.lp_begin = w.lp_begin;
  I.page_begin = w.page_begin;
  I.n_tiles = (w.n_pages + kTilePages - 1) / kTilePages;
  I.partial_begin = w.partial_begin;
  I.row_begin = w.row_begin;
  int col = 0;
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    I.rp[s] = 0; I.col[s] = col; I.pa[s] = 0; I.s[s] = 0.f; I.rc_off[s] = 0;
    const int ci = tile_agents[w.agent_begin + s];
    if (ci >= 0) {
      const int pa = ca[ci].pool_agent;
      const AgentDev dv = ag[pa];
      I.pa[s] = pa;
      I.rp[s] = dv.rp;
      I.s[s] = dv.s;
      I.rc_off[s] = dv.rc_off;
      col += dv.rp;
    }
  }
  I.sum_rp = col;
  I.n_groups = col / 8;
}

__device__ __forceinline__ uint32_t* err_word(const PoolGeom& g) {
  return (uint32_t*)(g.base + g.off_err);
}

// cos, sin of t * theta_i from the exact product of t with theta_i / 2 pi
// as a 64-bit fraction (the wrap modulo 2 pi is the integer overflow), so
// the hardware sine and cosine only ever see arguments in [-pi, pi].
__device__ __forceinline__ float2 rot_at(unsigned long long frac, int t) {
  const unsigned long long fr = (unsigned long long)(unsigned)t * frac;
  float ang = (float)(unsigned int)(fr >> 32) * 1.4629180792671596e-09f;   // 2 pi / 2^32
  if (ang > 3.14159265f) ang -= 6.28318531f;
  float sn, cs;
  __sincosf(ang, &sn, &cs);          // |ang| <= pi: absolute error ~4e-7, far below f16
  return make_float2(cs, sn);
}

// A zero the compiler cannot see through: mixed into values that would
// otherwise be hoisted out of a loop (descriptor sets, table conversions)
// and held in registers for all of it.
__device__ __forceinline__ uint32_t opaque_zero() {
  uint32_t z;
  asm volatile("mov.u32 %0, 0;" : "=r"(z));
  return z;
}

// A 16-byte read-only global load that stays where it is written: as
// volatile asm it is neither repeated at its point of use nor moved past
// the (volatile) tensor-memory waits around it, so its latency is spent
// while the warp does other work.
__device__ __forceinline__ uint4 ldg_pinned(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// M of one work item into shared memory, shared by the 384 threads of the
// compute and Trig warpgroups (bt = thread index among them).  Column
// n = 4 (8 j + e) + g for rank e of 8-rank group j and row g of the group's
// agent slot; feature 2i = s (q_i Bk[k,i] + q_{i+d/2} Bk[k,i+d/2]), feature
// 2i + 1 = s (q_{i+d/2} Bk[k,i] - q_i Bk[k,i+d/2]).  q is read from the
// staged Q rows (bf16), Bk from the pool (B-operand layout of Lk Bk).  A
// unit is (group j, frequency i, row g); the lane order (i % 4, g, i / 4)
// keeps the stores at most two-way bank conflicted.
__device__ __forceinline__ void build_m(const PoolGeom& g, int head, int n_groups, const Misc& Ms,
                                        uint8_t* smem, int layer, int bt) {
  constexpr int kBatch = 4;          // units whose Bk loads are in flight together
  const int n_units = n_groups * 4 * NF;
  const uint8_t* bk_base = g.base + g.off_bk + opaque_zero();   // not shared across the callers
  for (int u0 = bt; u0 < n_units; u0 += kBatch * 384) {
    uint4 b0[kBatch], b1[kBatch];
#pragma unroll
    for (int m = 0; m < kBatch; ++m) {
      const int u = u0 + m * 384;
      b0[m] = b1[m] = make_uint4(0, 0, 0, 0);
      if (u < n_units) {
        const int i = 4 * ((u >> 4) & 15) + (u & 3), j = u >> 8;
        const int s = Ms.mslot[j];
        const int RC = Ms.srp[s] / 8, kc = j - Ms.scol[s] / 8;
        const __nv_bfloat16* bk = (const __nv_bfloat16*)(bk_base + (int64_t)Ms.spa[s] * g.bk_agent_bytes) +
                                  ((int64_t)layer * g.H_kv + head) * (int64_t)D * g.rmax_pad;
        b0[m] = __ldg((const uint4*)(bk + ((i / 8) * RC + kc) * 64 + (i % 8) * 8));
        b1[m] = __ldg((const uint4*)(bk + (((i + NF) / 8) * RC + kc) * 64 + ((i + NF) % 8) * 8));
      }
    }
#pragma unroll
    for (int m = 0; m < kBatch; ++m) {
      const int u = u0 + m * 384;
      if (u < n_units) {
        const int i = 4 * ((u >> 4) & 15) + (u & 3), gq = (u >> 2) & 3, j = u >> 8;
        const int s = Ms.mslot[j];
        const float sa = Ms.ss[s];
        const int n = kRPA * s + gq;
        // q of row n, features i and i + d/2, from the Q rows' core matrices
        const uint8_t* qb = smem + oQ + (n / 8) * (D / 8) * 128 + (n % 8) * 16;
        const float x0 = sa * __bfloat162float(*(const __nv_bfloat16*)(qb + (i / 8) * 128 + (i % 8) * 2));
        const float x1 =
            sa * __bfloat162float(*(const __nv_bfloat16*)(qb + ((i + NF) / 8) * 128 + ((i + NF) % 8) * 2));
        const uint32_t w0[4] = {b0[m].x, b0[m].y, b0[m].z, b0[m].w};
        const uint32_t w1[4] = {b1[m].x, b1[m].y, b1[m].z, b1[m].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float bi = (e & 1) ? bf_hi(w0[e / 2]) : bf_lo(w0[e / 2]);
          const float bh = (e & 1) ? bf_hi(w1[e / 2]) : bf_lo(w1[e / 2]);
          *(uint32_t*)(smem + oM + ((4 * j + e / 2) * (D / 8) + i / 4) * 128 + (4 * (e & 1) + gq) * 16 +
                       (i % 4) * 4) = pack_h2(x0 * bi + x1 * bh, x1 * bi - x0 * bh);
        }
      }
    }
  }
}

// One 8-rank group j of a tile at this thread's key t: Z columns
// 4 (8 j + e) + g (v) against Lk[t, 8 j + e] (lkv, bf16), accumulated into
// the four rows of local slot `slot` (acc[4 slot + g]).
__device__ __forceinline__ void reduce_group(const uint4 lkv, const uint32_t (&v)[32], uint32_t slot,
                                             float (&acc)[16]) {
  const uint32_t lw[4] = {lkv.x, lkv.y, lkv.z, lkv.w};
  float t4[kRPA] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float l = (e & 1) ? bf_hi(lw[e / 2]) : bf_lo(lw[e / 2]);
    ffma2(t4[0], t4[1], l, l, __uint_as_float(v[e * kRPA]), __uint_as_float(v[e * kRPA + 1]));
    ffma2(t4[2], t4[3], l, l, __uint_as_float(v[e * kRPA + 2]), __uint_as_float(v[e * kRPA + 3]));
  }
  switch (slot) {
    case 0: acc[0] += t4[0]; acc[1] += t4[1]; acc[2] += t4[2]; acc[3] += t4[3]; break;
    case 1: acc[4] += t4[0]; acc[5] += t4[1]; acc[6] += t4[2]; acc[7] += t4[3]; break;
    case 2: acc[8] += t4[0]; acc[9] += t4[1]; acc[10] += t4[2]; acc[11] += t4[3]; break;
    default: acc[12] += t4[0]; acc[13] += t4[1]; acc[14] += t4[2]; acc[15] += t4[3]; break;
  }
}

// Trig row of key t (the f16 pairs [cos, sin](t th_i), i < 64) from the
// pool's table into registers: loaded a tile ahead, while the previous
// tile's Z MMAs still read the Trig columns; only the store waits for them.
__device__ __forceinline__ void load_trig(const uint8_t* table, int t, uint4 (&w)[NF / 4]) {
  const uint8_t* row = table + (int64_t)t * (NF * 4);
#pragma unroll
  for (int j = 0; j < NF / 4; ++j) w[j] = ldg_pinned(row + 16 * j);
}

__device__ __forceinline__ void store_trig(const uint4 (&w)[NF / 4], uint32_t taddr) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t a[16];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a[4 * e] = w[4 * q + e].x; a[4 * e + 1] = w[4 * q + e].y;
      a[4 * e + 2] = w[4 * q + e].z; a[4 * e + 3] = w[4 * q + e].w;
    }
    tmem_st16(taddr + 16 * q, a);
  }
}

}  // namespace d8

// Online-softmax max update of one compute warpgroup's 16 rows (rare: only
// when some row's tile max exceeds its running max by more than 2^8): new
// running maxima, rescale factors, and O^T, OL^T rescaled in TMEM.
static __device__ __forceinline__ void raise_max16(d8::Misc& M, const uint32_t (&sv)[16], int r0, int sw,
                                                int lane, int ln, int bar_sync, bool rescale,
                                                uint32_t t_o, uint32_t t_ol) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float v = __uint_as_float(sv[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) M.red[sw][r0 + j] = v;
  }
  named_bar(bar_sync, 128);
  if (ln < 16) {             // padded rows see only -inf: alpha stays 1
    const int j = r0 + ln;
    float al = 1.f;
    const float cm = fmaxf(fmaxf(M.red[0][j], M.red[1][j]), fmaxf(M.red[2][j], M.red[3][j]));
    const float mo = M.m_used[j];
    const float mn = fmaxf(mo, cm);
    if (mn > mo) { al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn); M.m_used[j] = mn; }
    M.alpha[j] = al;
  }
  named_bar(bar_sync, 128);
  if (rescale) {
    tc_fence_after();
    uint32_t raw[16];
    tmem_ld16_wait(t_o, raw);
#pragma unroll
    for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[r0 + e]);
    tmem_st16(t_o, raw);
    tmem_ld16_wait(t_ol, raw);
#pragma unroll
    for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[r0 + e]);
    tmem_st16(t_ol, raw);
    tmem_wait_st();
  }
}

__global__ void __launch_bounds__(d8::kThreads, 1)
    decode8_kernel(PoolGeom g, PlanDev p, int layer, const uint16_t* __restrict__ q) {
  using namespace d8;
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc& M = *reinterpret_cast<Misc*>(smem + oMISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* ws = g.base + g.off_ws;
  const int32_t* cta_items = (const int32_t*)(ws + p.off_cta);
  uint32_t* errw = err_word(g);
  volatile int* abort_flag = &M.abort_flag;
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&M.bar[i]); };
  uint64_t ph = kEmptyMask;          // parity each role waits for, bit i for barrier i
  auto wait = [&](int i) {
    uint32_t par = (uint32_t)(ph >> i) & 1u;
    const bool ok = mbar_wait_inl(bar(i), par, abort_flag, errw);
    ph ^= 1ull << i;
    return ok;
  };

  // ---- set-up: zero the page stages (rows past a ragged tile stay
  // finite) and the misc block, barriers, TMEM.
  // (M, Q and P are written in full before they are read; the page stages
  // keep stale but finite rows past a ragged last tile)
  for (int i = oKB + tid * 16; i < oQ; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  for (int i = oMISC + tid * 16; i < TOTAL; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), bar_count(i));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&M.tmem_base), 512);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_base;
  const int it_begin = cta_items[blockIdx.x], it_end = cta_items[blockIdx.x + 1];

  // Register split: the copy and MMA warpgroup hands registers to the
  // compute and Trig warpgroups; the shares add up to the launch's 512 x 128.
  // setmaxnreg.inc may only raise a warp's count and .dec only lower it
  // (the other direction is an illegal instruction), so each warpgroup's
  // direction follows from its share against the launch's 128.
  constexpr int kRegLow = 72, kRegCompute = 160, kRegTrig = 120;
  static_assert(128 * kRegLow + 256 * kRegCompute + 128 * kRegTrig == 65536, "register split");
  static_assert(kRegLow < 128 && kRegCompute > 128, "the copy/MMA warpgroup gives, the compute warpgroups take");
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegLow) : "memory");
    if (warp == 0 || warp == 3) {
      // ====================================== page copies (warps 0 and 3) ====
      // every lane waits; lane 0 posts the transaction count; the lanes then
      // split the tile's bulk copies (one page each).  Warp 0 copies keys,
      // warp 3 values; each runs ahead as far as its stage allows.
      const bool keys = warp == 0;
      const int b_full = keys ? B_KB_FULL : B_VB_FULL, b_empty = keys ? B_KB_EMPTY : B_VB_EMPTY;
      const uint32_t dst0 = sbase + (keys ? oKB : oVB);
      const uint8_t* region = g.base + (keys ? g.off_kb : g.off_vb) + (int64_t)layer * g.kb_layer_bytes;
      for (int it = it_begin; it < it_end; ++it) {
        const fk_work_item& w = ((const fk_work_item*)(ws + p.off_items))[it];
        const int n_pages = w.n_pages, head = w.head;
        const int n_tiles = (n_pages + kTilePages - 1) / kTilePages;
        const int32_t* pages = (const int32_t*)(ws + p.off_pages) + w.page_begin;
        // page id of this lane's page of the next tile, loaded a tile ahead
        int pg = lane < min(kTilePages, n_pages) ? pages[lane] : 0;
        // the key warp also prefetches the item's rCache rows into L2 a tile
        // ahead of the compute warps' Lk loads and the Trig warps' Lv loads:
        // lane s < 8 the Lk rows of slot s, lane 8 + s its Lv rows (one
        // contiguous block of rp x 256 bytes per 128-key tile)
        const uint8_t* pf = nullptr;
        int pf_rp = 0;
        const int t_item = w.lp_begin * kPage;
        auto prefetch_tile = [&](int k) {
          if (pf == nullptr || k >= n_tiles) return;
          const int t0 = t_item + k * kTileTok;
          const int nt = min(kTileTok, g.tcap - t0);
          if (nt > 0) bulk_prefetch_l2(pf + (int64_t)(t0 / 8) * pf_rp * 16, (uint32_t)((nt / 8) * pf_rp * 16));
        };
        for (int k = 0; k < n_tiles; ++k) {
          const int p0 = k * kTilePages;
          const int np = min(kTilePages, n_pages - p0);
          const int pg_k = pg;
          if (p0 + kTilePages + lane < n_pages && lane < kTilePages) pg = pages[p0 + kTilePages + lane];
          wait(b_empty);
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(b_full), np * PAGE_B);
          __syncwarp();
          if (lane < np && !*abort_flag)
            bulk_g2s(dst0 + lane * PAGE_B, region + ((int64_t)pg_k * g.H_kv + head) * PAGE_B, PAGE_B,
                     bar(b_full));
          if (keys) {
            if (k == 0 && lane < 2 * kSlots) {
              // (looked up once the first copies are on their way)
              const int ci = ((const int32_t*)(ws + p.off_tile_agents))[w.agent_begin + (lane & 7)];
              if (ci >= 0) {
                const int pa = ((const CallAgent*)(ws + p.off_call_agents))[ci].pool_agent;
                const AgentDev dv = ((const AgentDev*)(g.base + g.off_agents))[pa];
                pf_rp = dv.rp;
                pf = g.base + dv.rc_off + (int64_t)layer * rc_layer_bytes(g, dv.rp) +
                     (lane >= kSlots ? (int64_t)g.tcap * dv.rp * 2 : 0);
              }
              prefetch_tile(0);
            }
            prefetch_tile(k + 1);
          }
        }
      }
    } else if (warp == 1) {
      // ======================================= MMA issue (converged warp) ====
      const uint32_t id32 = idesc_f16(128, kRows, 1);
      int tc = 0;                      // tiles issued (all items), selects the P buffer
      for (int it = it_begin; it < it_end; ++it) {
        const fk_work_item& wi = ((const fk_work_item*)(ws + p.off_items))[it];
        const int n_tiles = (wi.n_pages + kTilePages - 1) / kTilePages;
        const int tc0 = tc;
        // base scores of the next tile into S (Kb landed, S released)
        auto issue_s = [&]() {
          tc_fence_after();
          __syncwarp();
          if (elect_one() && !*abort_flag) {
            const uint32_t sb = sbase + opaque_zero();
            const uint64_t dK = sdesc(sb + oKB, 128, (D / 8) * 128);
            const uint64_t dQ = sdesc(sb + oQ, 128, (D / 8) * 128);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_ss(tmem + kTmS, dK + (uint64_t)(ks * 16), dQ + (uint64_t)(ks * 16), id32,
                     ks > 0 ? 1u : 0u);
            mma_commit(bar(B_KB_EMPTY));
            mma_commit(bar(B_S_FULL));
          }
          __syncwarp();
        };
        // values of the item's tile j (global tile pt): O^T += Vb^T P (both
        // operands in shared memory), OL^T += Lv^T P (Lv^T in TMEM); P, Vb
        // and Lv^T are ready.  The two alternate, so that the shared-memory
        // and the tensor-memory operand reads overlap (measured faster than
        // running each accumulator's MMAs back to back).
        auto pv = [&](int j, int pt) {
          const int pb = pt & 1;
          tc_fence_after();
          __syncwarp();
          if (elect_one() && !*abort_flag) {
            const uint32_t sb = sbase + opaque_zero();
            const uint64_t dP = sdesc(sb + oP + pb * P_B, kPChunk, kPRowGroup);
            const uint64_t dV = sdesc(sb + oVB, (D / 8) * 128, 128);
#pragma unroll
            for (int ks = 0; ks < kTileTok / 16; ++ks) {
              const uint32_t acc = (j == 0 && ks == 0) ? 0u : 1u;
              const uint64_t bP = dP + (uint64_t)((ks * 2 * kPChunk) >> 4);
              mma_ss(tmem + kTmO, dV + (uint64_t)((ks * PAGE_B) >> 4), bP, id32, acc);
              mma_ts(tmem + kTmOL, tmem + kTmLv + 8 * ks, bP, id32, acc);
            }
            mma_commit(bar(B_VB_EMPTY));
            mma_commit(bar(B_LV_EMPTY));
            mma_commit(bar(B_PV_DONE0 + pb));
          }
          __syncwarp();
        };
        wait(B_Q_FULL);
        // the compute warps wrote the item's slot tables before Q_FULL
        const int ng0 = M.half_groups[0], ng1 = M.half_groups[1];
        const int nc0 = (ng0 + kZChunkGroups - 1) / kZChunkGroups;
        const int nc1 = (ng1 + kZChunkGroups - 1) / kZChunkGroups;
        // Z chunk m of warpgroup w: its 8-rank groups 4 m .. 4 m + 3 into
        // the warpgroup's buffer (the MMA warp has seen it free)
        auto issue_z = [&](int w, int m) {
          tc_fence_after();
          __syncwarp();
          if (elect_one() && !*abort_flag) {
            const int g0 = (w ? ng0 : 0) + kZChunkGroups * m;
            const int ng = min(kZChunkGroups, (w ? ng1 : ng0) - kZChunkGroups * m);
            const uint32_t idZ = idesc_f16(128, 32 * ng, 0);
            const uint64_t dM = sdesc(sbase + opaque_zero() + oM + g0 * 4 * (D / 8) * 128, 128, (D / 8) * 128);
            const uint32_t tA = tmem + kTmTrig;
            const uint32_t tD = tmem + tm_z(w);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_ts(tD, tA + 8 * ks, dM + (uint64_t)(ks * 16), idZ, ks > 0 ? 1u : 0u);
            mma_commit(bar(b_zf(w)));
          }
          __syncwarp();
        };
        // Issue order per tile k: the first Z chunk of each warpgroup (the
        // buffers were freed before the compute warps' softmax of tile
        // k - 1, so these run during it), the base scores of tile k + 1 (S
        // is free once the compute warps start tile k; the key stage
        // refills a tile ahead), the rest of Z(k) as the compute warps free
        // the buffers, then the values of tile k - 1, which run while the
        // compute warps read the last chunk and do their softmax (nothing
        // waits for them before tile k + 1).  The two warpgroups' chunks
        // alternate, so one warpgroup reads its chunk while the other's is
        // computed.
        auto z_chunks = [&](int m0, int m1) {
          for (int m = m0; m < m1; ++m) {
            if (m < nc0) { wait(b_ze(0)); issue_z(0, m); }
            if (m < nc1) { wait(b_ze(1)); issue_z(1, m); }
          }
        };
        const int ncm = max(nc0, nc1), nearly = min(1, ncm);
        wait(B_KB_FULL);
        wait(B_S_FREE);
        issue_s();
        wait(B_M_FULL);
        for (int k = 0; k < n_tiles; ++k) {
          wait(B_TRIG_FULL);
          z_chunks(0, nearly);
          if (k + 1 < n_tiles) {
            wait(B_KB_FULL);
            wait(B_S_FREE);
            issue_s();
          }
          z_chunks(nearly, ncm);
          if (elect_one()) mma_commit(bar(B_TRIG_EMPTY));   // every Z of the tile issued
          __syncwarp();
          if (k > 0) {
            wait(B_P_FULL0 + ((tc0 + k - 1) & 1));
            wait(B_VB_FULL);
            wait(B_LV_FULL);
            if (k == 1) wait(B_ACC_EMPTY);
            pv(k - 1, tc0 + k - 1);
          }
        }
        wait(B_P_FULL0 + ((tc0 + n_tiles - 1) & 1));
        wait(B_VB_FULL);
        wait(B_LV_FULL);
        if (n_tiles == 1) wait(B_ACC_EMPTY);
        pv(n_tiles - 1, tc0 + n_tiles - 1);
        tc = tc0 + n_tiles;
      }
      // drain: every MMA issued must complete before tensor memory is freed,
      // also after a timed-out wait (then no further MMA was issued)
      if (elect_one()) mma_commit(bar(B_FINAL));
      __syncwarp();
      mbar_wait_drain(bar(B_FINAL), 0);
    }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegCompute) : "memory");
    // ====================================== compute warpgroups (4-11) ====
    const int cw = (warp - 4) >> 2;                  // warpgroup 0 or 1
    const int ln = 32 * (warp & 3) + lane;           // TMEM lane = key / d / rank slot
    const int sw = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int bar_sync = 1 + 2 * cw, bar_or = 2 + 2 * cw;   // this warpgroup's named barriers
    const int r0 = 16 * cw;                          // first query row of this warpgroup
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)D);
    const int32_t* row_agent_all = (const int32_t*)(ws + p.off_row_agent);
    const int32_t* row_cg_all = (const int32_t*)(ws + p.off_row_cg);
    const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
    int tc = 0, pv_seen = 0;
    // The value MMAs of tile j signal PV_DONE[j & 1].  Alternating barriers
    // keep a waiter within one phase of each, which parity waits need.
    auto pv_until = [&](int n) {
      while (pv_seen < n) { wait(B_PV_DONE0 + (pv_seen & 1)); ++pv_seen; }
    };
    for (int it = it_begin; it < it_end; ++it) {
      Item I;
      load_item(g, p, ws, it, I);
      // ---- item set-up.  Every MMA that read the previous item's Q and M
      // has completed (the Trig warps wait for the last Z commit of an item
      // before they join the M build below, and the last S of an item comes
      // before its last Z), so both may be rewritten once the named barrier
      // with the Trig warps has passed.
      named_bar(bar_sync, 128);                 // this warpgroup is done with the tables
      // 8-rank groups of this warpgroup's slots (an unrolled select: indexing
      // the record by the runtime warpgroup number would move it to local
      // memory)
      const int g_lo = (cw ? I.col[4] : I.col[0]) / 8;
      const int g_hi = cw ? I.sum_rp / 8 : I.col[4] / 8;
      {
        const int32_t* row_agent = row_agent_all + I.row_begin;
        const int32_t* row_cg = row_cg_all + I.row_begin;
        if (ln < 16) {
          const int j = r0 + ln;
          M.m_used[j] = -INFINITY;
          int lim = 0;
          const int ci = row_agent[j];
          if (ci >= 0) {
            const int T = ca[ci].seq_len;
            lim = p.causal ? min(T, T - p.C + row_cg[j] / g.G + 1) : T;
          }
          M.row_lim[j] = lim;
        }
        if (ln == 0) {
          int mn = 0x7fffffff;
          for (int j = r0; j < r0 + 16; ++j) {
            const int ci = row_agent[j];
            if (ci < 0) { mn = 0; break; }      // padded rows must stay masked
            const int T = ca[ci].seq_len;
            mn = min(mn, p.causal ? min(T, T - p.C + row_cg[j] / g.G + 1) : T);
          }
          M.lim_min[cw] = mn;
        }
        // Lk group tables of this warpgroup's slots; the tile's group owners
        if (ln < kWGGroups) {
          const int jl = ln, j = g_lo + jl;
          M.gbase[cw][jl] = nullptr;
          M.gstride[cw][jl] = 0;
          M.gslot[cw][jl] = 0;
#pragma unroll
          for (int s = 0; s < kSlots; ++s)
            if (j < g_hi && 8 * j >= I.col[s] && 8 * j < I.col[s] + I.rp[s]) {
              M.gbase[cw][jl] = g.base + I.rc_off[s] + (int64_t)layer * rc_layer_bytes(g, I.rp[s]) +
                                (int64_t)((8 * j - I.col[s]) / 8) * 128;
              M.gstride[cw][jl] = I.rp[s] * 16;
              M.gslot[cw][jl] = s - 4 * cw;
            }
        }
        if (cw == 0 && ln < kMaxGroups) {
          int os = 0;
#pragma unroll
          for (int s = 0; s < kSlots; ++s)
            if (8 * ln >= I.col[s] && 8 * ln < I.col[s] + I.rp[s]) os = s;
          M.mslot[ln] = os;
        }
        if (cw == 0 && ln < kSlots) {
#pragma unroll
          for (int s = 0; s < kSlots; ++s)
            if (s == ln) {
              M.srp[s] = I.rp[s]; M.scol[s] = I.col[s]; M.spa[s] = I.pa[s];
              M.ss[s] = I.s[s]; M.src[s] = I.rc_off[s];
            }
          if (ln == 0) { M.half_groups[0] = I.col[4] / 8; M.half_groups[1] = (I.sum_rp - I.col[4]) / 8; }
        }
        // Q rows r0 .. r0 + 15 (bf16, B operand of the base scores)
        for (int u = ln; u < 16 * (D / 8); u += 128) {
          const int row = r0 + u / (D / 8), ch = u % (D / 8);
          uint4 v = make_uint4(0, 0, 0, 0);
          const int ci = row_agent[row];
          if (ci >= 0) {
            const int cg = row_cg[row];
            const int64_t qrow = ((int64_t)ci * p.C + cg / g.G) * g.H_q + I.head * g.G + cg % g.G;
            v = *(const uint4*)(q + qrow * D + ch * 8);
          }
          *(uint4*)(smem + oQ + ((row / 8) * (D / 8) + ch) * 128 + (row % 8) * 16) = v;
        }
      }
      fence_proxy_async();
      named_bar(bar_sync, 128);                 // tables visible to the whole warpgroup
      if (lane == 0) mbar_arrive(bar(B_Q_FULL));
      named_bar(5, 384);                        // every Q row staged: build M
      build_m(g, I.head, I.n_groups, M, smem, layer, tid - 128);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_M_FULL));

      // Lk of this thread's key, loaded into registers a tile ahead: the
      // loads of tile k + 1 are issued once tile k's Z reduction has used
      // the registers (a lane past the rCache capacity reads the last row:
      // its key is masked)
      uint4 lk[kWGGroups];
#pragma unroll
      for (int jl = 0; jl < kWGGroups; ++jl) lk[jl] = make_uint4(0, 0, 0, 0);
      {
        const int t = min(I.lp_begin * kPage + ln, g.tcap - 1);
#pragma unroll
        for (int jl = 0; jl < kWGGroups; ++jl)
          if (g_lo + jl < g_hi)
            lk[jl] = ldg_pinned(M.gbase[cw][jl] + (int64_t)(t / 8) * M.gstride[cw][jl] + (t % 8) * 16);
      }
      // OL^T lane ln: rank orr of the slot os whose columns hold ln (that
      // slot's rows take it in the epilogue)
      int os = -1, orr = 0;
#pragma unroll
      for (int s = 0; s < kSlots; ++s)
        if (ln >= I.col[s] && ln < I.col[s] + I.rp[s]) { os = s; orr = ln - I.col[s]; }
      uint32_t gsl = 0;                // 4 bits per local group: its slot in the warpgroup
#pragma unroll
      for (int jl = 0; jl < kWGGroups; ++jl) gsl |= (uint32_t)M.gslot[cw][jl] << (4 * jl);
      // this lane's share of row (lane / 2)'s sum of P over the tiles (the
      // running maxima are read from shared memory, where only raise_max16
      // changes them)
      float l_acc = 0.f;

      for (int k = 0; k < I.n_tiles; ++k, ++tc) {
        const int t0 = (I.lp_begin + k * kTilePages) * kPage;
        const int ntok = min(kTileTok, (I.n_pages - k * kTilePages) * kPage);
        // base scores of rows r0 .. r0 + 15: S(k) was issued before Z(k), so
        // the first Z chunk's commit covers it
        uint32_t sv[16];
        wait(B_S_FULL);
        tc_fence_after();
        tmem_ld16_wait(tmem + kTmS + r0 + lane_off, sv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(bar(B_S_FREE));
        // residual scores: acc[4 s + g] += sum_e Lk[t, 8 j + e] Z[t, 4 (8 j + e) + g]
        // for the 8-rank groups j of local slot s.  This warpgroup's chunk m
        // holds its local groups 4 m .. 4 m + 3.
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll
        for (int jl = 0; jl < kWGGroups; ++jl) {
          if (g_lo + jl < g_hi) {
            if (jl % kZChunkGroups == 0) {
              wait(b_zf(cw));
              tc_fence_after();
            }
            uint32_t v[32];
            tmem_ld32_wait(tmem + tm_z(cw) + 32 * (jl % kZChunkGroups) + lane_off, v);
            // chunk read: the MMA may overwrite the buffer
            if (jl % kZChunkGroups == kZChunkGroups - 1 || g_lo + jl + 1 >= g_hi) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_relaxed(bar(b_ze(cw)));
            }
            reduce_group(lk[jl], v, (gsl >> (4 * jl)) & 3u, acc);
          }
        }
        // Lk of the next tile (after the TMEM loads above, whose waits must
        // not cover these)
        if (k + 1 < I.n_tiles) {
          const int tn = min((I.lp_begin + (k + 1) * kTilePages) * kPage + ln, g.tcap - 1);
#pragma unroll
          for (int jl = 0; jl < kWGGroups; ++jl)
            if (g_lo + jl < g_hi)
              lk[jl] = ldg_pinned(M.gbase[cw][jl] + (int64_t)(tn / 8) * M.gstride[cw][jl] + (tn % 8) * 16);
        }
        // ---- online softmax (base 2); the running max of a row moves only
        // when the tile max exceeds it by more than 2^8 (then O^T, OL^T and
        // the row sums are rescaled)
        // (the rows' running maxima and limits are read into registers
        // first, in 16-byte loads: loads from shared memory interleaved with
        // the stores of P below would be kept in program order)
        float mv[16];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(&M.m_used[r0 + j]);
          mv[j] = m4.x; mv[j + 1] = m4.y; mv[j + 2] = m4.z; mv[j + 3] = m4.w;
        }
        bool need = false;
        if (ntok == kTileTok && t0 + kTileTok <= M.lim_min[cw]) {
          // every key of the tile is visible to every row of this warpgroup
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float s = (__uint_as_float(sv[j]) + acc[j]) * scale_log2;
            sv[j] = __float_as_uint(s);
            need |= s > mv[j] + 8.f;
          }
        } else {
          const int tabs = t0 + ln;
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const int4 l4 = *reinterpret_cast<const int4*>(&M.row_lim[r0 + j]);
            const int lim[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool ok = ln < ntok && tabs < lim[u];
              const float s = ok ? (__uint_as_float(sv[j + u]) + acc[j + u]) * scale_log2 : -INFINITY;
              sv[j + u] = __float_as_uint(s);
              need |= s > mv[j + u] + 8.f;
            }
          }
        }
        int any;
        asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, 128, p; selp.u32 %0, 1, 0, q; }"
                     : "=r"(any) : "r"((int)need), "r"(bar_or));
        if (any) {
          if (k > 0) pv_until(tc);           // O^T, OL^T hold every earlier tile
          raise_max16(M, sv, r0, sw, lane, ln, bar_sync, k > 0, tmem + kTmO + r0 + lane_off,
                      tmem + kTmOL + r0 + lane_off);
          l_acc *= M.alpha[r0 + (lane >> 1)];
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(&M.m_used[r0 + j]);
            mv[j] = m4.x; mv[j + 1] = m4.y; mv[j + 2] = m4.z; mv[j + 3] = m4.w;
          }
        }
        // P of this tile into P buffer tc & 1 (its previous reader is PV(tc - 2))
        pv_until(tc - 1);
        uint8_t* prow = smem + oP + (tc & 1) * P_B + (r0 / 8) * kPRowGroup + (ln / 8) * kPChunk + (ln % 8) * 2;
        float rs[16];
        uint16_t pbits[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float m = mv[j];
          // 2^x of x <= 8 (or -inf): the hardware approximation, far finer
          // than the bf16 rounding that follows
          float pe;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pe) : "f"(__uint_as_float(sv[j]) - (m == -INFINITY ? 0.f : m)));
          const __nv_bfloat16 pb = __float2bfloat16_rn(pe);
          pbits[j] = *reinterpret_cast<const uint16_t*>(&pb);
          rs[j] = __bfloat162float(pb);       // row sums of the same rounded P
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) *(uint16_t*)(prow + (j / 8) * kPRowGroup + (j % 8) * 16) = pbits[j];
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL0 + (tc & 1)));
        // row sums over this warp's 32 keys: a reduce-scatter that leaves
        // row (lane / 2)'s sum in lanes lane & ~1 and lane | 1
#pragma unroll
        for (int h = 8; h >= 1; h >>= 1) {
          const bool up = (lane & (2 * h)) != 0;   // keep the upper half of the rows
#pragma unroll
          for (int i = 0; i < h; ++i) {
            const float send = up ? rs[i] : rs[i + h];
            const float keep = up ? rs[i + h] : rs[i];
            rs[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * h);
          }
        }
        l_acc += rs[0] + __shfl_xor_sync(0xffffffffu, rs[0], 1);
      }
      // ---- epilogue: this warpgroup's rows of the item's split partials
      pv_until(tc);
      tc_fence_after();
      if ((lane & 1) == 0) M.red[sw][r0 + (lane >> 1)] = l_acc;
      named_bar(bar_sync, 128);
      {
        const int32_t* row_agent = row_agent_all + I.row_begin;
        float* part = (float*)(ws + p.off_partials);
        const int PS = p.partial_stride;
        uint32_t raw[16];
        tmem_ld16_wait(tmem + kTmO + r0 + lane_off, raw);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (row_agent[r0 + e] >= 0)
            part[(int64_t)(I.partial_begin + r0 + e) * PS + 4 + ln] = __uint_as_float(raw[e]);
        tmem_ld16_wait(tmem + kTmOL + r0 + lane_off, raw);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = r0 + e;
          if (os >= 0 && row / kRPA == os && row_agent[row] >= 0)
            part[(int64_t)(I.partial_begin + row) * PS + 4 + D + orr] = __uint_as_float(raw[e]);
        }
        if (ln < 16 && row_agent[r0 + ln] >= 0) {
          float* dst = part + (int64_t)(I.partial_begin + r0 + ln) * PS;
          dst[0] = M.m_used[r0 + ln];
          dst[1] = M.red[0][r0 + ln] + M.red[1][r0 + ln] + M.red[2][r0 + ln] + M.red[3][r0 + ln];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(bar(B_ACC_EMPTY));
    }
  } else {
    if constexpr (kRegTrig > 128)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegTrig) : "memory");
    else if constexpr (kRegTrig < 128)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegTrig) : "memory");
    // ======================================== Trig and Lv^T (warps 12-15) ====
    // Trig column i of a tile holds [cos, sin]((t0 + lane) theta_i) as an
    // f16 pair, copied from the pool's table of per-position rotations.
    // Tile k + 1's Trig is loaded into registers a tile ahead and stored
    // once Z(k) has completed.  Lv^T: lane = rank slot of the tile; 16 loads
    // of 8 keys each, stored as bf16 key pairs once the value MMAs of the
    // previous tile have completed.
    const uint8_t* trig_table = g.base + g.off_trig;
    const int ln = 32 * (warp & 3) + lane;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    int zdone = 0;                    // tiles whose Z MMAs are known complete
    auto z_until = [&](int n) {
      while (zdone < n) { wait(B_TRIG_EMPTY); ++zdone; }
    };
    // (no closure refers to the loaded Trig: an array captured by
    // reference stays in local memory)
    auto trig_full = [&]() {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(bar(B_TRIG_FULL));
    };
    int tc = 0;
    for (int it = it_begin; it < it_end; ++it) {
      const fk_work_item& wi = ((const fk_work_item*)(ws + p.off_items))[it];
      const int head = wi.head, n_tiles = (wi.n_pages + kTilePages - 1) / kTilePages;
      const int tb = wi.lp_begin * kPage;
      // M may be rewritten once every Z of the previous item has completed
      z_until(tc);
      named_bar(5, 384);                        // the compute warps staged Q and the slot tables
      build_m(g, head, wi.sum_rank / 8, M, smem, layer, tid - 128);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_M_FULL));
      // this lane's rank slot of the tile: Lv of 8 keys at
      // lvp + (t / 8) * lvs (lanes past the tile's ranks store zeros)
      const uint8_t* lvp = nullptr;
      int64_t lvs = 0;
      for (int s = 0; s < kSlots; ++s)
        if (ln >= M.scol[s] && ln < M.scol[s] + M.srp[s]) {
          const int r = ln - M.scol[s], rp = M.srp[s];
          lvp = g.base + M.src[s] + (int64_t)layer * rc_layer_bytes(g, rp) +
                (int64_t)g.tcap * rp * 2 + (r / 8) * 128 + (r % 8) * 16;
          lvs = (int64_t)rp * 16;
        }
      // half hh of tile k's Lv^T (keys 64 hh .. 64 hh + 63): eight loads of
      // 8 keys each, stored as 32 columns of bf16 key pairs
      auto lv_half = [&](int k, int hh) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int ch = min(tb / 8 + 16 * k + 8 * hh + c, g.tcap / 8 - 1);
          const uint4 v = lvp ? __ldg((const uint4*)(lvp + (int64_t)ch * lvs)) : make_uint4(0, 0, 0, 0);
          w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
        // the first half's loads are in flight while the previous tile's
        // value MMAs finish with Lv^T
        if (hh == 0) wait(B_LV_EMPTY);
        tc_fence_after();
        tmem_st32(tmem + kTmLv + 32 * hh + lane_off, w);
      };
      // (keys past the capacity are masked; they read the last row)
      uint4 tw[NF / 4];
      load_trig(trig_table, min(tb + ln, g.tcap - 1), tw);
      store_trig(tw, tmem + kTmTrig + lane_off);
      trig_full();
      if (n_tiles > 1) load_trig(trig_table, min(tb + kTileTok + ln, g.tcap - 1), tw);
      for (int k = 0; k < n_tiles; ++k) {
        // Trig of tile k + 1 (loaded a tile ahead), stored once Z(k) has
        // completed; then the load of tile k + 2's, and Lv^T of tile k (free
        // once the value MMAs of tile k - 1 have completed)
        if (k + 1 < n_tiles) {
          z_until(tc + k + 1);
          tc_fence_after();
          store_trig(tw, tmem + kTmTrig + lane_off);
          trig_full();
          if (k + 2 < n_tiles) load_trig(trig_table, min(tb + (k + 2) * kTileTok + ln, g.tcap - 1), tw);
        }
        lv_half(k, 0);
        lv_half(k, 1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(bar(B_LV_FULL));
      }
      tc += n_tiles;
    }
    z_until(tc);
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

// ============================================================ RoPE table ==

// [cos, sin](t theta_i) as f16 pairs for t < tcap, i < 64: one thread per
// element, from the exact phase (the same rotation the oracle rounds).
__global__ void trig_table_kernel(PoolGeom g) {
  const int64_t n = (int64_t)g.tcap * d8::NF;
  const unsigned long long* frac = (const unsigned long long*)(g.base + g.off_rope + 256);
  uint32_t* table = (uint32_t*)(g.base + g.off_trig);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / d8::NF), i = (int)(e % d8::NF);
    const float2 r = d8::rot_at(frac[i], t);
    table[e] = pack_h2(r.x, r.y);
  }
}

int launch_trig_table(const PoolGeom& g) {
  if (g.off_trig < 0 || g.d != d8::D) return (int)cudaErrorInvalidValue;
  const int64_t n = (int64_t)g.tcap * d8::NF;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  trig_table_kernel<<<grid, 256>>>(g);
  return (int)cudaGetLastError();
}

// ============================================================ launcher ==

bool decode8_applies(const PoolGeom& g, const PlanDev& p) {
  return p.slots8 != 0 && g.d == d8::D && g.G * p.C == d8::kRPA;
}

int launch_decode8(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q, void* stream) {
  static PerDeviceOnce once;
  const int se = once.run([] {
    cudaError_t e = cudaFuncSetAttribute(decode8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, d8::TOTAL);
    if (e != cudaSuccess) return (int)e;
    // the warps' register split (setmaxnreg) hands out exactly the block's
    // launch registers, 512 x 128: a build with another count would leave
    // the compute warps waiting for registers, so it is refused here
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, decode8_kernel);
    if (e != cudaSuccess) return (int)e;
    return fa.numRegs == 128 ? 0 : (int)cudaErrorInvalidConfiguration;
  });
  if (se != 0) return se;
  decode8_kernel<<<p.n_ctas, d8::kThreads, d8::TOTAL, (cudaStream_t)stream>>>(g, p, layer, q);
  return (int)cudaGetLastError();
}

}  // namespace fk
