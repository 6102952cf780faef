// Residual attention for decode-shaped work tiles (four query rows per
// agent, e.g. one decode query of a GQA group of four heads).
//
// The scores of agent a at key position t are (ForkKV guide,
// "Mathematical Formulation of ResidualAttention")
//     q . (Kb[t] + s RoPE_t(Lk[t] Bk)) / sqrt(d).
// RoPE is linear and acts per frequency pair (i, i + d/2), so the residual
// term regroups as
//     q . RoPE_t(Lk[t] Bk) = sum_k Lk[t,k] Z[t,(k,g)],
//     Z[t,(k,g)] = sum_i cos(t th_i) Mc[i,(k,g)] + sin(t th_i) Ms[i,(k,g)],
//     Mc = q_i Bk[k,i] + q_{i+d/2} Bk[k,i+d/2],
//     Ms = q_{i+d/2} Bk[k,i] - q_i Bk[k,i+d/2].
// Z is one dense contraction per 128-key tile, Trig(t) [128 x d] times
// M [d x 4 r] (M built once per work item from Bk and the queries), run on
// the tensor cores with N = 4 r; the length-r sum against Lk[t] runs on the
// CUDA cores next to the softmax.  Compared with rebuilding
// RoPE(Lk Bk) for every key and agent and contracting it with four query
// rows, this issues a quarter of the MMA instructions (each N = 16 MMA
// costs as much tensor-pipe time as an N = 96 one on GB300) and replaces
// the d-wide RoPE pass by an r-wide dot product.
//
// The value residual keeps its factored form (LRAgent summary, section 3):
// O^T = Vb^T P and OL^T = [Lv | 1]^T P on the tensor cores, Bv applied once
// per row in the combine.  Partials and the combine are shared with the
// general kernel.
//
// M is built per (agent tile, kv head) by a small preceding grid straight
// into the workspace in the kernel's shared-memory image (the kernel starts
// under programmatic dependent launch and waits for that grid only before
// its first copy of M).
//
// Warp roles (512 threads): warp 0 key (and M) bulk copies, warp 3 value
// copies, warp 1 MMA issue (converged warp, elect.sync), warp 2 dequantiser
// of the compressed pool; warps 4-7 and 8-11 two compute warpgroups;
// warps 12-15 the Trig warpgroup.  Compute warpgroup w owns query rows
// 8w .. 8w+7 (agents 2w, 2w+1): their Z reduction, online softmax, P and
// epilogue.  The Trig warpgroup writes each tile's Trig two tiles ahead.
// setmaxnreg moves registers from the copy, MMA and Trig warps to the
// compute warpgroups.  A warp reaches TMEM lanes 32 (warp % 4) .. +31, so
// a thread of TMEM lane 32 (warp % 4) + lane handles the key (or d, or
// rank) of that lane.
#include <cuda_runtime.h>

#include <cstdint>

#include "fk_device.cuh"
#include "fk_internal.h"
#include "fk_once.h"

namespace fk {
namespace dec {

constexpr int kThreads = 512;       // 16 warps
constexpr int kRPA = 4;               // query rows per agent
constexpr int kRows = 16;             // padded query rows of a tile (<= 4 agents)
constexpr int kA = kMaxAgentsPerTile;
constexpr int kMaxZ = kRPA * kMaxRankSum;   // Z columns of a tile: (rank, row) pairs
constexpr int kZBuf = 128;            // Z columns per TMEM buffer
constexpr int kPChunk = 144;          // P: 8 keys x 8 rows core matrix, padded
constexpr int kPRowGroup = 16 * kPChunk;
// [Lv | 1]^T stage: rank group m (8 ranks x 128 keys, 16 core matrices of
// 8 ranks x 8 keys) at m * kLvGroup; groups 0-7 hold the tile's agents'
// ranks in column order, group 8 the ones row (TMEM lane 64 of OL^T)
constexpr int kLvGroup = 16 * 128;
constexpr int kOnesLane = 64;
// TMEM columns: base scores (two buffers of 16 rows: 0 and 48), O^T, OL^T
// (16 rows each), two Trig stages (64 and 192), the per-lane rotation
// table, two Z buffers (one per 128-column chunk of a tile's Z)
constexpr uint32_t kTmS = 0, kTmOT = 16, kTmOL = 32, kTmS1 = 48, kTmTrig0 = 64, kTmTau = 128,
                   kTmTrig1 = 192, kTmZ = 256;
__host__ __device__ constexpr uint32_t tm_s(int b) { return b ? kTmS1 : kTmS; }
__host__ __device__ constexpr uint32_t tm_trig(int b) { return b ? kTmTrig1 : kTmTrig0; }

template <int D, bool COMP>
struct Layout {
  static constexpr int PAGE_B = kPage * D * 2;
  static constexpr int TILE_B = kTilePages * PAGE_B;
  static constexpr int NKB = 2;
  static constexpr int NVB = COMP ? 1 : 2;
  static constexpr int M_B = (kMaxZ / 8) * (D / 8) * 128;
  static constexpr int LV_B = 9 * kLvGroup;
  static constexpr int Q_B = kRows * D * 2;
  static constexpr int P_B = 2 * kPRowGroup;
  static constexpr int KQ_B = COMP ? kTilePages * kPage * D : 0;
  // compressed values: two stages of codes and norms, so that the value
  // warp copies tile k + 1's while it expands tile k's
  static constexpr int VCS_B = kTilePages * kPage * (3 * D / 8);
  static constexpr int VNS_B = kTilePages * kPage * 4;
  static constexpr int VC_B = COMP ? 2 * VCS_B : 0;
  static constexpr int VN_B = COMP ? 2 * VNS_B : 0;
  static constexpr int oM = 0;
  static constexpr int oKB = oM + M_B;
  static constexpr int oVB = oKB + NKB * TILE_B;   // d = 64: the Vb^T MMA reads 1 KB past a stage
  static constexpr int oLV = oVB + NVB * TILE_B;   // the OL^T MMA (M = 128) reads 16 groups
  static constexpr int oQ = oLV + LV_B;            // from here: lanes 72-127 are never used
  static constexpr int oP = oQ + Q_B;                // two P buffers
  static constexpr int oKQ = oP + 2 * P_B;
  static constexpr int oVC = oKQ + KQ_B;
  static constexpr int oVN = oVC + VC_B;
  static constexpr int oMISC = (oVN + VN_B + 127) / 128 * 128;
  static constexpr int MISC_B = 4096;
  static constexpr int TOTAL =
      (oMISC + MISC_B > oLV + 16 * kLvGroup) ? oMISC + MISC_B : oLV + 16 * kLvGroup;
};

enum {
  B_KB_FULL0, B_KB_FULL1, B_KB_EMPTY0, B_KB_EMPTY1, B_VB_FULL0, B_VB_FULL1, B_VB_EMPTY0,
  B_VB_EMPTY1, B_LV_FULL, B_LV_EMPTY, B_M_FULL, B_M_EMPTY, B_ITEM_FULL, B_TRIG_FULL0, B_TRIG_FULL1, B_Z_FULL0, B_Z_FULL1, B_Z_FREE0, B_Z_FREE1, B_P_FULL0, B_P_FULL1, B_PV_DONE0,
  B_PV_DONE1, B_ACC_EMPTY, B_KQ_FULL, B_KQ_EMPTY, B_VC_FULL0, B_VC_FULL1, B_VC_EMPTY0, B_VC_EMPTY1,
  B_FINAL,
  B_STALL,   // never completed: the target of the failure-detection test's wait
  B_COUNT
};
// Arrival counts: 8 = lane 0 of each warp of both compute warpgroups; 4 =
// lane 0 of each Trig warp; 1 = one thread, a bulk-copy transaction count
// or an MMA commit.
__host__ __device__ constexpr uint32_t bar_count(int i) {
  return (i == B_ITEM_FULL || i == B_Z_FREE0 || i == B_Z_FREE1 || i == B_P_FULL0 ||
          i == B_P_FULL1 || i == B_ACC_EMPTY)
             ? 8u
             : (i == B_TRIG_FULL0 || i == B_TRIG_FULL1) ? 4u : 1u;
}
// compressed pool: the value stage is filled by two warps (0 and 3), each
// expanding half of a tile's code units
template <bool COMP>
__host__ __device__ constexpr uint32_t bar_count_t(int i) {
  return (COMP && (i == B_VB_FULL0 || i == B_VB_FULL1)) ? 2u : bar_count(i);
}
constexpr uint64_t kEmptyMask =
    (1ull << B_KB_EMPTY0) | (1ull << B_KB_EMPTY1) | (1ull << B_VB_EMPTY0) | (1ull << B_VB_EMPTY1) |
    (1ull << B_LV_EMPTY) | (1ull << B_M_EMPTY) | (1ull << B_Z_FREE0) | (1ull << B_Z_FREE1) |
    (1ull << B_ACC_EMPTY) | (1ull << B_KQ_EMPTY) | (1ull << B_VC_EMPTY0) | (1ull << B_VC_EMPTY1);
static_assert(B_COUNT <= 64, "one parity bit per barrier");

struct Misc {
  uint64_t bar[B_COUNT];
  uint32_t tmem_base;
  int abort_flag;
  float m_used[kRows];
  float alpha[kRows];
  float red[4][kRows];
  int32_t row_lim[kRows];          // key t is visible to row j iff t < row_lim[j]
  int32_t lim_min[2];              // smallest row_lim of each warpgroup's rows (0: padded rows)
  float2 rot[4][64];               // per Trig warp: cos, sin of t0 * theta_i of the
                                   // tile being written
  unsigned long long frac[64];     // theta_i / (2 pi) as a 64-bit binary fraction
  // per compute warpgroup and 8-rank group j: owning agent (0 or 1 within the
  // warpgroup) and the address of key t's 8 ranks,
  // gbase + (t / 8) * gstride + (t % 8) * 16
  const uint8_t* gbase[2][8];
  int32_t gstride[2][8];
  int32_t gagent[2][8];
  // the dequantiser's copy of the 3-bit value codebook: lanes index it with
  // their own codes, which a constant-memory table would serve one address
  // at a time
  float lloyd[8];
};
static_assert(sizeof(Misc) <= 4096, "Misc must fit its smem slot");

struct Item {
  int head, n_rows, n_pages, lp_begin, n_ag, partial_begin, n_tiles, page_begin, sum_rp, next;
  int rp[kA], col[kA], pool_agent[kA];
  // Lv^T stage columns: agents that read the same residual rows (Shared-A:
  // LRAgent summary, "BaseLRShared") share one block, copied once, and one
  // OL^T rank block serves all of their rows; lv_rp = the stage's ranks
  int lvcol[kA], lv_rp;
  float s[kA];
  int64_t rc_off[kA];
};

// Work item `it` of this call (records 0 .. gridDim.x - 1 are the CTAs'
// first items; `next` chains the rest), looked up by the host.
__device__ __forceinline__ const DecItem* ditem(const PlanDev& p, const uint8_t* ws, int it) {
  return (const DecItem*)(ws + p.off_ditems) + it;
}

__device__ __forceinline__ void load_item(const PlanDev& p, const uint8_t* ws, int it, Item& I) {
  const DecItem& w = *ditem(p, ws, it);
  I.head = w.head;
  I.n_rows = w.n_rows;
  I.n_pages = w.n_pages;
  I.lp_begin = w.lp_begin;
  I.n_ag = w.n_ag;
  I.partial_begin = w.partial_begin;
  I.page_begin = w.page_begin;
  I.sum_rp = w.sum_rp;
  I.next = w.next;
  I.lv_rp = w.lv_rp;
  I.n_tiles = (w.n_pages + kTilePages - 1) / kTilePages;
#pragma unroll
  for (int a = 0; a < kA; ++a) {
    I.rp[a] = w.rp[a];
    I.col[a] = w.col[a];
    I.pool_agent[a] = w.pool_agent[a];
    I.lvcol[a] = w.lvcol[a];
    I.s[a] = w.s[a];
    I.rc_off[a] = w.rc_off[a];
  }
}

__device__ __forceinline__ const uint8_t* rc_lk(const PoolGeom& g, const Item& I, int a, int layer) {
  return g.base + I.rc_off[a] + (int64_t)layer * rc_layer_bytes(g, I.rp[a]);
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

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace dec

// Online-softmax max update of one compute warpgroup's 8 rows (rare: only
// when some row's tile max exceeds its running max by more than 2^8): new
// running maxima, rescale factors, and O^T, OL^T rescaled in TMEM.  Kept out
// of line so the tile loop stays small.
static __device__ __noinline__ void raise_max(dec::Misc& M, uint32_t s0, uint32_t s1, uint32_t s2,
                                              uint32_t s3, uint32_t s4, uint32_t s5, uint32_t s6,
                                              uint32_t s7, int r0, int sw, int lane, int ln,
                                              int bar_sync, bool rescale, uint32_t t_ot,
                                              uint32_t t_ol) {
  const uint32_t sv[8] = {s0, s1, s2, s3, s4, s5, s6, s7};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float v = __uint_as_float(sv[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) M.red[sw][r0 + j] = v;
  }
  named_bar(bar_sync, 128);
  if (ln < 8) {             // padded rows see only -inf: alpha stays 1
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
    uint32_t raw[8];
    tmem_ld8_wait(t_ot, raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[r0 + e]);
    tmem_st8(t_ot, raw);
    tmem_ld8_wait(t_ol, raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[r0 + e]);
    tmem_st8(t_ol, raw);
    tmem_wait_st();
  }
}

template <int D, bool COMP>
__global__ void __launch_bounds__(dec::kThreads, 1)
    decode_kernel(PoolGeom g, PlanDev p, int layer, const uint16_t* __restrict__ q) {
  using namespace dec;
  using LY = Layout<D, COMP>;
  constexpr int NF = D / 2;                  // RoPE frequencies
  constexpr int SBO_M = (D / 8) * 128;       // M: K-major core matrices, features along K
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc& M = *reinterpret_cast<Misc*>(smem + LY::oMISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* ws = g.base + g.off_ws;
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
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- set-up: zero smem (rows the padded MMAs read stay finite), the
  // ones row of the Lv^T stage, RoPE fractions, barriers, TMEM.
  for (int i = tid * 16; i < LY::TOTAL; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int i = tid; i < 16 * 8; i += kThreads)
    ((uint16_t*)(smem + LY::oLV + (kOnesLane / 8) * kLvGroup + (i / 8) * 128))[i % 8] = 0x3F80;
  if (tid < 64) M.frac[tid] = ((const unsigned long long*)(g.base + g.off_rope + 256))[tid];
  if (COMP && tid < 8) M.lloyd[tid] = c_lloyd[tid];
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), bar_count_t<COMP>(i));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&M.tmem_base), 512);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_base;

  // Register split: the copy and MMA warps (warpgroup 0) and the Trig
  // warpgroup hand registers to the two compute warpgroups; the shares add
  // up to the launch's 512 x 128 (the dequantiser of the compressed pool
  // keeps more in warpgroup 0).
  constexpr int kRegCopy = COMP ? 120 : 104, kRegTrig = 88, kRegCompute = COMP ? 152 : 160;
  static_assert(128 * kRegCopy + 128 * kRegTrig + 256 * kRegCompute <= 65536, "register split");
  // Compressed pool: half `half` of global tile vt's code units (np pages)
  // -> level * norm / D in the value layout (rotated domain).  A unit is
  // (page, 8-token chunk, 8-d group): three code bytes per token, one per
  // bit plane.  Warp 0 expands half 0 and frees the code stage; warp 3 (the
  // stage's copier, which reads it in program order) expands half 1.  Both
  // arrive on the value stage's full barrier (count 2).
  auto expand_values = [&](int np, int vt, int half) {
    const int cst = vt & 1;
    wait(B_VC_FULL0 + cst);
    wait(B_VB_EMPTY0);
    uint8_t* vdst = smem + LY::oVB;
    const uint8_t* vc = smem + LY::oVC + cst * LY::VCS_B;
    const float* vn = (const float*)(smem + LY::oVN + cst * LY::VNS_B);
    const uint8_t* book = (const uint8_t*)M.lloyd;
    for (int u = lane + 32 * half; u < np * 2 * (D / 8); u += 64) {
      const int dg = u % (D / 8), tcn = (u / (D / 8)) % 2, pj = u / (2 * (D / 8));
      float w8[8];
      uint32_t c8[8];
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        const int row = tcn * 8 + tt;
        const uint8_t* cb = vc + (pj * kPage + row) * (3 * D / 8);
        const uint32_t b0 = cb[dg], b1 = cb[D / 8 + dg], b2 = cb[2 * (D / 8) + dg];
        // bit e of the planes at bits e + 2, e + 11, e + 20: shifted right
        // by e, e + 8, e + 16 and masked, a code's bits give its byte
        // offset (4 x code) into the codebook
        c8[tt] = (b0 << 2) | (b1 << 11) | (b2 << 20);
        w8[tt] = vn[pj * kPage + row] * (1.0f / D);
      }
      uint8_t* dst = vdst + pj * LY::PAGE_B + (tcn * (D / 8) + dg) * 128;
      // each lane writes the 8 rows of its core in its own rotation, so that
      // the lanes of one store hit different banks
#pragma unroll
      for (int s8 = 0; s8 < 8; ++s8) {
        const int e = (s8 + lane) & 7;   // d = 8 dg + e
        uint32_t w[4];
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
          float v2[2];
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            const uint32_t cc = c8[2 * h2 + z];
            const uint32_t off = ((cc >> e) & 4u) | ((cc >> (8 + e)) & 8u) | ((cc >> (16 + e)) & 16u);
            v2[z] = *(const float*)(book + off) * w8[2 * h2 + z];
          }
          w[h2] = pack_bf2(v2[0], v2[1]);
        }
        *(uint4*)(dst + e * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bar(B_VB_FULL0));
      if (half == 0) mbar_arrive(bar(B_VC_EMPTY0 + cst));
    }
  };
  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegCopy) : "memory");
  if (warp == 0) {
    // ============================================== key copies (warp 0) ====
    // every lane waits; lane 0 posts the transaction count; the lanes then
    // split the tile's bulk copies (one page each).  Keys run ahead as far as
    // the two key stages allow, independently of the values.
    // (failure-detection test: a wait that gives up, so that the whole CTA
    // takes its abort path and the call reports the timeout)
    if (p.stall_probe) wait(B_STALL);
    int tc = 0;
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      Item I;
      load_item(p, ws, it, I);
      if (I.n_pages == 0) break;   // a CTA without work
      nxt = I.next;
      const int32_t* pages = (const int32_t*)(ws + p.off_pages) + I.page_begin;
      const int tc0 = tc;
      // page id of this lane's page of the next tile, loaded a tile ahead
      // (the first tile's come with the item)
      int pg = lane < kTilePages ? ditem(p, ws, it)->first_pages[lane] : 0;
      for (int k = 0; k < I.n_tiles; ++k) {
        const int p0 = k * kTilePages;
        const int np = min(kTilePages, I.n_pages - p0);
        const int pg_k = pg;
        if (p0 + kTilePages + lane < I.n_pages && lane < kTilePages) pg = pages[p0 + kTilePages + lane];
        tc = tc0 + k;
        if (!COMP) {
          const int st = tc & 1;
          wait(B_KB_EMPTY0 + st);
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_KB_FULL0 + st), np * LY::PAGE_B);
          __syncwarp();
          if (lane < np && !*abort_flag) {
            const uint8_t* src = g.base + g.off_kb + (int64_t)layer * g.kb_layer_bytes +
                                 ((int64_t)pg_k * g.H_kv + I.head) * LY::PAGE_B;
            bulk_g2s(sbase + LY::oKB + st * LY::TILE_B + lane * LY::PAGE_B, src, LY::PAGE_B,
                     bar(B_KB_FULL0 + st));
          }
        } else {
          wait(B_KQ_EMPTY);
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_KQ_FULL), np * kPage * D);
          __syncwarp();
          if (lane < np && !*abort_flag) {
            const uint8_t* src = g.base + g.off_kq +
                                 ((((int64_t)layer * g.num_pages + pg_k) * g.H_kv + I.head) * kPage) * D;
            bulk_g2s(sbase + LY::oKQ + lane * kPage * D, src, kPage * D, bar(B_KQ_FULL));
          }
        }
        if (k == 0) {
        // the item's M (built by the preceding grid) once the previous item's
        // Z MMAs are done with the buffer; after the first key tile, which
        // need not wait for that
        {
          const DecItem* rec = ditem(p, ws, it);
          const uint32_t mbytes = (uint32_t)rec->mbytes;
          const uint8_t* msrc = ws + rec->mofs;
          wait(B_M_EMPTY);
          if (it == (int)blockIdx.x) asm volatile("griddepcontrol.wait;" ::: "memory");
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_M_FULL), mbytes);
          __syncwarp();
          for (uint32_t o = lane * 4096u; o < mbytes && !*abort_flag; o += 32u * 4096u)
            bulk_g2s(sbase + LY::oM + o, msrc + o, min(4096u, mbytes - o), bar(B_M_FULL));
        }
        }
        // compressed pool: half of the previous tile's values
        if (COMP && k > 0) expand_values(min(kTilePages, I.n_pages - (k - 1) * kTilePages), tc - 1, 0);
      }
      if (COMP) expand_values(min(kTilePages, I.n_pages - (I.n_tiles - 1) * kTilePages), tc0 + I.n_tiles - 1, 0);
      tc = tc0 + I.n_tiles;
    }
  } else if (warp == 3) {
    // ============================================= value copies (warp 3) ====
    // values of tile k: Vb (or the compressed codes) and the Lv^T stage
    int tc = 0;
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      Item I;
      load_item(p, ws, it, I);
      if (I.n_pages == 0) break;   // a CTA without work
      nxt = I.next;
      const int32_t* pages = (const int32_t*)(ws + p.off_pages) + I.page_begin;
      // page id of this lane's page of the next tile, loaded a tile ahead
      // (the first tile's come with the item)
      int pg = lane < kTilePages ? ditem(p, ws, it)->first_pages[lane] : 0;
      auto load_values = [&](int k, int vt) {
        const int p0 = k * kTilePages;
        const int np = min(kTilePages, I.n_pages - p0);
        const int t0 = (I.lp_begin + p0) * kPage;
        const int pg_k = pg;
        if (p0 + kTilePages + lane < I.n_pages && lane < kTilePages) pg = pages[p0 + kTilePages + lane];
        if (COMP) {
          // codes and norms into stage vt & 1 (this warp expanded its
          // previous contents, tile vt - 2, before the proxy fence that ends
          // that expansion)
          const int cst = vt & 1;
          wait(B_VC_EMPTY0 + cst);   // warp 0 has expanded its half of tile vt - 2
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_VC_FULL0 + cst), np * kPage * (3 * D / 8 + 4));
          __syncwarp();
          if (lane < np && !*abort_flag) {
            const int64_t tok = (((int64_t)layer * g.num_pages + pg_k) * g.H_kv + I.head) * kPage;
            bulk_g2s(sbase + LY::oVC + cst * LY::VCS_B + lane * kPage * (3 * D / 8),
                     g.base + g.off_vc + tok * (3 * D / 8), kPage * (3 * D / 8), bar(B_VC_FULL0 + cst));
            bulk_g2s(sbase + LY::oVN + cst * LY::VNS_B + lane * kPage * 4, g.base + g.off_vn + tok * 4,
                     kPage * 4, bar(B_VC_FULL0 + cst));
          }
          // then the previous tile's values are expanded, before the Lv^T
          // copy below waits for the value MMAs that consume them
          if (k > 0) expand_values(min(kTilePages, I.n_pages - (k - 1) * kTilePages), vt - 1, 1);
        } else {
          const int st = vt % LY::NVB;
          wait(B_VB_EMPTY0 + st);
          __syncwarp();
          if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_VB_FULL0 + st), np * LY::PAGE_B);
          __syncwarp();
          if (lane < np && !*abort_flag) {
            const uint8_t* src = g.base + g.off_vb + (int64_t)layer * g.kb_layer_bytes +
                                 ((int64_t)pg_k * g.H_kv + I.head) * LY::PAGE_B;
            bulk_g2s(sbase + LY::oVB + st * LY::TILE_B + lane * LY::PAGE_B, src, LY::PAGE_B,
                     bar(B_VB_FULL0 + st));
          }
        }
        // Lv^T: one tensor copy per rank group of each distinct rCache block
        // (its agent's Lv map, coordinates (0, 0, group, t0 / 8, layer)) into
        // group lvcol / 8 + j
        wait(B_LV_EMPTY);
        const int n_grp = I.lv_rp / 8;
        __syncwarp();
        if (lane == 0 && !*abort_flag) mbar_expect_tx_relaxed(bar(B_LV_FULL), n_grp * kLvGroup);
        __syncwarp();
        if (lane < n_grp && !*abort_flag) {
          int pa = 0, j = 0;
#pragma unroll
          for (int a = 0; a < kA; ++a)
            if (a < I.n_ag && lane >= I.lvcol[a] / 8 && lane < (I.lvcol[a] + I.rp[a]) / 8) {
              pa = I.pool_agent[a];
              j = lane - I.lvcol[a] / 8;
            }
          const uint8_t* map = g.base + g.off_lvmap + 128LL * pa;
          asm volatile(
              "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
              " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(sbase + LY::oLV + lane * kLvGroup),
              "l"(map), "r"(0), "r"(0), "r"(j), "r"(t0 / 8), "r"(layer), "r"(bar(B_LV_FULL))
              : "memory");
        }
      };
      for (int k = 0; k < I.n_tiles; ++k, ++tc) load_values(k, tc);
      if (COMP) expand_values(min(kTilePages, I.n_pages - (I.n_tiles - 1) * kTilePages), tc - 1, 1);
    }
  } else if (warp == 1) {
    // ======================================= MMA issue (converged warp) ====
    const uint32_t idS = idesc_f16(128, kRows, 1);
    int tc = 0;
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      Item I;
      load_item(p, ws, it, I);
      if (I.n_pages == 0) break;   // a CTA without work
      nxt = I.next;
      const int zcols = kRPA * I.sum_rp;
      const int n_zc = (zcols + kZBuf - 1) / kZBuf;
      wait(B_M_FULL);                    // the item's M
      wait(B_ITEM_FULL);                 // its Q, row tables, first Trig stages
      tc_fence_after();
      // values of tile j (global tile pt): O^T += Vb^T P, OL^T += [Lv | 1]^T P,
      // both A operands in shared memory
      auto pv = [&](int j, int pt) {
        const int pb = pt & 1, vs = pt % LY::NVB;
        wait(B_P_FULL0 + pb);
        wait(B_VB_FULL0 + vs);
        wait(B_LV_FULL);
        if (j == 0) wait(B_ACC_EMPTY);
        tc_fence_after();
        __syncwarp();
        if (elect_one() && !*abort_flag) {
          const uint64_t dP = sdesc(sbase + LY::oP + pb * LY::P_B, kPChunk, kPRowGroup);
          const uint64_t dV = sdesc(sbase + LY::oVB + vs * LY::TILE_B, (D / 8) * 128, 128);
          const uint64_t dL = sdesc(sbase + LY::oLV, 128, kLvGroup);
#pragma unroll
          for (int ks = 0; ks < kTileTok / 16; ++ks) {
            const uint32_t acc = (j == 0 && ks == 0) ? 0u : 1u;
            const uint64_t bP = dP + (uint64_t)((ks * 2 * kPChunk) >> 4);
            mma_ss(tmem + kTmOT, dV + (uint64_t)((ks * LY::PAGE_B) >> 4), bP, idS, acc);
            mma_ss(tmem + kTmOL, dL + (uint64_t)((ks * 256) >> 4), bP, idS, acc);
          }
          mma_commit(bar(B_VB_EMPTY0 + vs));
          mma_commit(bar(B_LV_EMPTY));
          mma_commit(bar(B_PV_DONE0 + pb));
        }
        __syncwarp();
      };
      // base scores of global tile t into S buffer t & 1.  Its previous
      // reader, tile t - 2, released it with Z_FREE0 (the compute warpgroups
      // read S before the first Z chunk), which this warp has waited for.
      // The Z_FULL commits of tile t cover these MMAs.
      auto issue_s = [&](int t) {
        const int kb = t & 1;
        wait(B_KB_FULL0 + kb);
        tc_fence_after();
        __syncwarp();
        if (elect_one() && !*abort_flag) {
          const uint64_t dK = sdesc(sbase + LY::oKB + kb * LY::TILE_B, 128, (D / 8) * 128);
          const uint64_t dQ = sdesc(sbase + LY::oQ, 128, (D / 8) * 128);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss(tmem + tm_s(kb), dK + (uint64_t)(ks * 16), dQ + (uint64_t)(ks * 16), idS,
                   ks > 0 ? 1u : 0u);
          mma_commit(bar(B_KB_EMPTY0 + kb));
        }
        __syncwarp();
      };
      // per tile k: Z(k) chunk by chunk (Trig(k) was written two tiles
      // ahead; chunk c waits for the reads of chunk c of tile k - 1), the
      // values of tile k - 1, which wait for that tile's P, then the next
      // tile's base scores, whose keys get the longest lead this way.
      const int tc0 = tc;
      issue_s(tc0);
      for (int k = 0; k < I.n_tiles; ++k) {
        tc = tc0 + k;
        const int st = tc & 1;
        wait(B_TRIG_FULL0 + st);
        for (int c = 0; c < n_zc; ++c) {
          wait(B_Z_FREE0 + c);
          tc_fence_after();
          __syncwarp();
          if (elect_one() && !*abort_flag) {
            const int ncol = min(kZBuf, zcols - c * kZBuf);
            const uint32_t idZ = idesc_f16(128, ncol, 0);
            const uint64_t dM = sdesc(sbase + LY::oM + c * (kZBuf / 8) * SBO_M, 128, SBO_M);
            const uint32_t tA = tmem + tm_trig(st);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_ts(tmem + kTmZ + c * kZBuf, tA + 8 * ks, dM + (uint64_t)(ks * 16), idZ,
                     ks > 0 ? 1u : 0u);
            mma_commit(bar(B_Z_FULL0 + c));
          }
          __syncwarp();
        }
        if (k > 0) pv(k - 1, tc - 1);
        if (k + 1 < I.n_tiles) issue_s(tc + 1);
      }
      if (elect_one()) mma_commit(bar(B_M_EMPTY));   // every Z MMA of the item is issued
      __syncwarp();
      pv(I.n_tiles - 1, tc0 + I.n_tiles - 1);
      tc = tc0 + I.n_tiles;
    }
    // drain: every MMA issued must complete before tensor memory is freed,
    // also after a timed-out wait (then no further MMA was issued)
    if (elect_one()) mma_commit(bar(B_FINAL));
    __syncwarp();
    mbar_wait_drain(bar(B_FINAL), 0);
  } else if (COMP && warp == 2) {
    // ====================================== dequantiser (compressed pool) ====
    const float kscale = ((const float*)(g.base + g.off_ks))[layer];
    int tc = 0;
    // keys only: the value warp expands the values
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      Item I;
      load_item(p, ws, it, I);
      if (I.n_pages == 0) break;   // a CTA without work
      nxt = I.next;
      const int tc0 = tc;
      for (int j = 0; j < I.n_tiles; ++j) {
        {
          const int k = j;
          const int np = min(kTilePages, I.n_pages - k * kTilePages);
          const int kb = (tc0 + k) & 1;
          // keys: int8 [page][16][D] -> bf16 (value * scale) in the key layout
          wait(B_KQ_FULL);
          wait(B_KB_EMPTY0 + kb);
          uint8_t* kdst = smem + LY::oKB + kb * LY::TILE_B;
          // lanes take the 8 rows of a core matrix first, so that a warp's
          // 16-byte stores fill whole 128-byte cores (no bank conflicts)
          for (int u = lane; u < np * kPage * (D / 8); u += 32) {
            const int ch = (u / 8) % (D / 8), row = (u % 8) + 8 * ((u / (8 * (D / 8))) % 2),
                      pj = u / (kPage * (D / 8));
            // eight int8 keys in one 8-byte load
            const uint2 kw = *(const uint2*)(smem + LY::oKQ + (pj * kPage + row) * D + ch * 8);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t src = e < 2 ? kw.x : kw.y;
              const int sh = 16 * (e & 1);
              w[e] = pack_bf2((float)(int8_t)(src >> sh) * kscale, (float)(int8_t)(src >> (sh + 8)) * kscale);
            }
            *(uint4*)(kdst + pj * LY::PAGE_B + ((row / 8) * (D / 8) + ch) * 128 + (row % 8) * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) { mbar_arrive(bar(B_KB_FULL0 + kb)); mbar_arrive(bar(B_KQ_EMPTY)); }
        }
      }
      tc = tc0 + I.n_tiles;
    }
  }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegCompute) : "memory");
    // ====================================== compute warpgroups (4-11) ====
    const int cw = (warp - 4) >> 2;                  // warpgroup 0 or 1
    const int ln = 32 * (warp & 3) + lane;           // TMEM lane = key / d / rank
    const int sw = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int bar_sync = 1 + 2 * cw, bar_or = 2 + 2 * cw;   // this warpgroup's named barriers
    const int r0 = 8 * cw;                           // first query row of this warpgroup
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)D);
    int tc = 0, pv_seen = 0;
    // The value MMAs of tile j signal PV_DONE[j & 1].  Alternating barriers
    // keep a waiter within one phase of each, which parity waits need.
    auto pv_until = [&](int n) {
      while (pv_seen < n) { wait(B_PV_DONE0 + (pv_seen & 1)); ++pv_seen; }
    };
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      int n_tiles, lp_begin, n_pages, n_zc, g_lo, g_hi;
      bool split;
      // ---- item set-up.  Every MMA that read the previous item's Q and
      // Trig stages has completed (this warpgroup waited for all of them:
      // the Z_FULL commits of a tile cover its S MMAs), so those buffers are
      // free without a barrier of their own.
      named_bar(bar_sync, 128);                 // this warpgroup is done with the tables
      {
        Item I;
        load_item(p, ws, it, I);
        if (I.n_pages == 0) break;              // a CTA without work
        nxt = I.next;
        const DecItem* rec = ditem(p, ws, it);
        const int n_rows = I.n_rows, n_ag = I.n_ag;
        n_tiles = I.n_tiles;
        lp_begin = I.lp_begin;
        n_pages = I.n_pages;
        n_zc = (kRPA * I.sum_rp + kZBuf - 1) / kZBuf;
        // (an unrolled select: indexing the record by the runtime warpgroup
        // number would move it to local memory)
        const int c_lo = cw ? I.col[2] : I.col[0], c_hi = cw ? I.sum_rp : I.col[2];
        g_lo = c_lo / 8;
        g_hi = c_hi / 8;
        // split item: every row is warpgroup 0's (one or two agents), and
        // warpgroup 1 takes the upper half of the rank groups; it hands its
        // sums for warpgroup 0's rows over each tile
        split = rec->split != 0;
        if (split) {
          const int G = I.sum_rp / 8, gm = (G + 1) / 2;
          g_lo = cw ? gm : 0;
          g_hi = cw ? G : gm;
        }
        // rows: limits and running maxima
        if (ln < 8) {
          const int j = r0 + ln;
          M.m_used[j] = -INFINITY;
          M.row_lim[j] = rec->row_lim[j];
        }
        if (ln == 0) M.lim_min[cw] = rec->lim_min[cw];
        // Lk group tables of this warpgroup's agents
        if (ln < 8) {
          const int j = ln;
          int aj = 0;
#pragma unroll
          for (int a = 1; a < kA; ++a)
            if (a < n_ag && 8 * j >= I.col[a]) aj = a;
          M.gagent[cw][j] = aj - (split ? 0 : 2 * cw);
          M.gbase[cw][j] = nullptr;
          M.gstride[cw][j] = 0;
#pragma unroll
          for (int a = 0; a < kA; ++a)
            if (a == aj && j >= g_lo && j < g_hi) {
              M.gbase[cw][j] = rc_lk(g, I, a, layer) + (int64_t)((8 * j - I.col[a]) / 8) * 128;
              M.gstride[cw][j] = I.rp[a] * 16;
            }
        }
        // Q rows r0 .. r0 + 7 (bf16, B operand of the base scores)
        for (int u = ln; u < 8 * (D / 8); u += 128) {
          const int row = r0 + u / (D / 8), ch = u % (D / 8);
          uint4 v = make_uint4(0, 0, 0, 0);
          const int qrow = row < n_rows ? rec->qrow[row] : -1;
          if (qrow >= 0) v = *(const uint4*)(q + (int64_t)qrow * D + ch * 8);
          *(uint4*)(smem + LY::oQ + ((row / 8) * (D / 8) + ch) * 128 + (row % 8) * 16) = v;
        }
        fence_proxy_async();
        named_bar(bar_sync, 128);               // tables visible to the whole warpgroup
        if (lane == 0) mbar_arrive(bar(B_ITEM_FULL));
      }
      // Lk of this thread's key, loaded into registers a tile ahead: the
      // loads of tile k + 1 are issued once tile k's Z reduction has used
      // the registers, so they arrive while this tile finishes
      uint4 lkA[4] = {}, lkB[4] = {};  // rank groups 0-3 and 4-7 (two arrays: the chunk
                                       // select below stays a register select)
      // (a lane past the rCache capacity reads the last row instead: its
      // key is masked; registers of groups this warpgroup does not own keep
      // stale values and are never read, so no load result is merged with a
      // constant, which would make the issue wait for the load)
      auto load_lk = [&](int k) {
        const int t = min((lp_begin + k * kTilePages) * kPage + ln, g.tcap - 1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j >= g_lo && j < g_hi)
            lkA[j] = __ldg((const uint4*)(M.gbase[cw][j] + (int64_t)(t / 8) * M.gstride[cw][j] + (t % 8) * 16));
          if (j + 4 >= g_lo && j + 4 < g_hi)
            lkB[j] = __ldg((const uint4*)(M.gbase[cw][j + 4] + (int64_t)(t / 8) * M.gstride[cw][j + 4] + (t % 8) * 16));
        }
      };
      load_lk(0);
      uint32_t gmask = 0;              // bit j: rank group j belongs to this warpgroup's second agent
#pragma unroll
      for (int j = 0; j < 8; ++j) gmask |= (M.gagent[cw][j] == 1) ? (1u << j) : 0u;
      // running maxima of this warpgroup's rows, kept in registers (the
      // shared copy changes only in raise_max)
      float mreg[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mreg[j] = -INFINITY;

      for (int k = 0; k < n_tiles; ++k, ++tc) {
        const int t0 = (lp_begin + k * kTilePages) * kPage;
        const int ntok = min(kTileTok, (n_pages - k * kTilePages) * kPage);
        // base scores of rows r0 .. r0 + 7: S(k) was issued before Z(k), so
        // the first Z chunk's commit covers it
        uint32_t sv[8];
        wait(B_Z_FULL0);
        tc_fence_after();
        tmem_ld8_wait(tmem + tm_s(tc & 1) + r0 + lane_off, sv);
        // residual scores: acc[4 la + g] = sum_k Lk[t,k] Z[t,(col + k) * 4 + g]
        // for local agent la of this warpgroup
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 1
        for (int c = 0; c < n_zc; ++c) {
          if (c > 0) {
            wait(B_Z_FULL0 + c);
            tc_fence_after();
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * c + u;      // 8-rank group of these 32 columns
            if (j >= g_lo && j < g_hi) {
              const uint4 L = c ? lkB[u] : lkA[u];
              const uint32_t lw[4] = {L.x, L.y, L.z, L.w};
              float t4[kRPA] = {0.f, 0.f, 0.f, 0.f};
              uint32_t v[32];
              tmem_ld32_wait(tmem + kTmZ + c * kZBuf + 32 * u + lane_off, v);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float l = (e & 1) ? bf_hi(lw[e / 2]) : bf_lo(lw[e / 2]);
                ffma2(t4[0], t4[1], l, l, __uint_as_float(v[e * kRPA]), __uint_as_float(v[e * kRPA + 1]));
                ffma2(t4[2], t4[3], l, l, __uint_as_float(v[e * kRPA + 2]), __uint_as_float(v[e * kRPA + 3]));
              }
              const bool second = (gmask >> j) & 1u;
#pragma unroll
              for (int gq = 0; gq < kRPA; ++gq) {
                acc[gq] += second ? 0.f : t4[gq];
                acc[kRPA + gq] += second ? t4[gq] : 0.f;
              }
            }
          }
          // chunk c (and, for c = 0, the S buffer) read: Z(k + 1) chunk c
          // and S(k + 2) may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(bar(B_Z_FREE0 + c));
        }
        if (split) {
          // warpgroup 1's sums of warpgroup 0's rows, handed over through
          // the S columns of warpgroup 1's own rows (padded in a split
          // item, and already read): warp w and warp w + 4 reach the same
          // TMEM lanes.  The buffer's next S comes after both warpgroups
          // have released this tile's first Z chunk.  Both warpgroups wait
          // at the barrier, so each of its phases is one tile's hand-off
          // (with an arrive-only producer a phase could also complete on
          // two of the producer's arrivals).
          const uint32_t xcol = tmem + tm_s(tc & 1) + 8 + lane_off;
          uint32_t xw[8];
          if (cw == 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) xw[j] = __float_as_uint(acc[j]);
            tmem_st8(xcol, xw);
            tmem_wait_st();
            tc_fence_before();
            named_bar(6, 256);
          } else {
            named_bar(6, 256);
            tc_fence_after();
            tmem_ld8_wait(xcol, xw);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += __uint_as_float(xw[j]);
          }
        }
        if (k + 1 < n_tiles) load_lk(k + 1);
        // ---- online softmax (base 2); the running max of a row moves only
        // when the tile max exceeds it by more than 2^8 (then O^T, OL^T are
        // rescaled in TMEM)
        bool need = false;
        if (ntok == kTileTok && t0 + kTileTok <= M.lim_min[cw]) {
          // every key of the tile is visible to every row of this warpgroup
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float s = (__uint_as_float(sv[j]) + acc[j]) * scale_log2;
            sv[j] = __float_as_uint(s);
            need |= s > mreg[j] + 8.f;
          }
        } else {
          const int tabs = t0 + ln;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const bool ok = ln < ntok && tabs < M.row_lim[r0 + j];
            const float s = ok ? (__uint_as_float(sv[j]) + acc[j]) * scale_log2 : -INFINITY;
            sv[j] = __float_as_uint(s);
            need |= s > mreg[j] + 8.f;
          }
        }
        int any;
        asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, 128, p; selp.u32 %0, 1, 0, q; }"
                     : "=r"(any) : "r"((int)need), "r"(bar_or));
        if (any) {
          if (k > 0) pv_until(tc);           // O^T, OL^T hold every earlier tile
          raise_max(M, sv[0], sv[1], sv[2], sv[3], sv[4], sv[5], sv[6], sv[7], r0, sw, lane, ln,
                    bar_sync, k > 0, tmem + kTmOT + r0 + lane_off, tmem + kTmOL + r0 + lane_off);
#pragma unroll
          for (int j = 0; j < 8; ++j) mreg[j] = M.m_used[r0 + j];
        }
        // P of this tile into P buffer tc & 1 (its previous reader is PV(tc - 2))
        pv_until(tc - 1);
        uint8_t* prow = smem + LY::oP + (tc & 1) * LY::P_B + cw * kPRowGroup + (ln / 8) * kPChunk + (ln % 8) * 2;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float m = mreg[j];
          // 2^x of x <= 8 (or -inf): the hardware approximation, far finer
          // than the bf16 rounding that follows
          float pv;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(pv) : "f"(__uint_as_float(sv[j]) - (m == -INFINITY ? 0.f : m)));
          *(__nv_bfloat16*)(prow + j * 16) = __float2bfloat16_rn(pv);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL0 + (tc & 1)));

      }
      // ---- epilogue: this warpgroup's rows of the item's split partials
      pv_until(tc);
      tc_fence_after();
      {
        Item I;
        load_item(p, ws, it, I);
        const int n_rows = I.n_rows, n_ag = I.n_ag;
        float* part = (float*)(ws + p.off_partials);
        const int PS = p.partial_stride;
        uint32_t raw[8];
        tmem_ld8_wait(tmem + kTmOT + r0 + lane_off, raw);
        if (ln < D) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (r0 + e < n_rows) part[(int64_t)(I.partial_begin + r0 + e) * PS + 4 + ln] = __uint_as_float(raw[e]);
        }
        // OL^T lane ln: for each row, rank ln - lvcol of the row's agent if
        // its Lv block holds ln (a shared block serves every agent reading
        // it), or the row sums on the ones lane
        tmem_ld8_wait(tmem + kTmOL + r0 + lane_off, raw);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int row = r0 + e;
          // the row's agent, 2 cw + e / 4, as an unrolled select
          const int la = cw ? I.lvcol[2 + e / 4] : I.lvcol[e / 4];
          const int lr = cw ? I.rp[2 + e / 4] : I.rp[e / 4];
          if (row < n_rows) {
            float* dst = part + (int64_t)(I.partial_begin + row) * PS;
            if (ln == kOnesLane) dst[1] = __uint_as_float(raw[e]);
            if (row / kRPA < n_ag && ln >= la && ln < la + lr) dst[4 + D + ln - la] = __uint_as_float(raw[e]);
          }
        }
        if (ln < 8 && r0 + ln < n_rows) part[(int64_t)(I.partial_begin + r0 + ln) * PS] = M.m_used[r0 + ln];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(bar(B_ACC_EMPTY));
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegTrig) : "memory");
    // ======================================== Trig tiles (warps 12-15) ====
    // Trig column i of a tile holds [cos, sin]((t0 + lane) theta_i) as an
    // f16 pair: the tile start's rotation (exact phase, computed by each
    // warp for itself, one frequency per lane) composed in fp32 with the
    // rotation of the lane's key offset tau, a table kept in TMEM.  Tile
    // k's Trig goes to stage (global tile) & 1, written once the Z MMAs of
    // tile k - 2 (the stage's last readers) have completed.
    const int ln = 32 * (warp & 3) + lane;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll 1
    for (int c0 = 0; c0 < NF; c0 += 16) {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 r = rot_at(M.frac[c0 + e], ln);
        w[e] = pack_h2(r.x, r.y);
      }
      tmem_st16(tmem + kTmTau + c0 + lane_off, w);
    }
    tmem_wait_st();
    float2* rotw = M.rot[warp - 12];
    auto make_trig = [&](int t0, int st) {
      for (int f = lane; f < NF; f += 32) rotw[f] = rot_at(M.frac[f], t0);
      __syncwarp();
#pragma unroll 1
      for (int c0 = 0; c0 < NF; c0 += 16) {
        uint32_t w[16];
        tmem_ld16_wait(tmem + kTmTau + c0 + lane_off, w);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 rb = rotw[c0 + e];
          const float2 rt = __half22float2(as_h2(w[e]));
          w[e] = pack_h2(rb.x * rt.x - rb.y * rt.y, rb.y * rt.x + rb.x * rt.y);
        }
        tmem_st16(tmem + tm_trig(st) + c0 + lane_off, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();                             // rotw readers done before the next write
      if (lane == 0) mbar_arrive_relaxed(bar(B_TRIG_FULL0 + st));
    };
    int tc = 0;
    for (int it = (int)blockIdx.x, nxt; it >= 0; it = nxt) {
      Item I;
      load_item(p, ws, it, I);
      if (I.n_pages == 0) break;   // a CTA without work
      nxt = I.next;
      const int n_zc = (kRPA * I.sum_rp + kZBuf - 1) / kZBuf;
      const int tb = I.lp_begin * kPage;
      make_trig(tb, tc & 1);
      if (I.n_tiles > 1) make_trig(tb + kTileTok, (tc + 1) & 1);
      for (int k = 0; k < I.n_tiles; ++k, ++tc) {
        for (int c = 0; c < n_zc; ++c) wait(B_Z_FULL0 + c);   // Z(k) has completed
        tc_fence_after();
        if (k + 2 < I.n_tiles) make_trig(tb + (k + 2) * kTileTok, tc & 1);
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

// ============================================================= M build ==
// M of one (agent tile, kv head) pair, in the decode kernel's shared-memory
// image: column n = (col[a] + k) * 4 + row-in-agent, K-major core matrices
// of 8 columns x 8 features, feature 2i the cos part, 2i + 1 the sin part,
// times s_a.  One thread per unit = (8-rank group j, row gq of the agent,
// frequency i): two 16-byte loads of Bk (ranks 8j.. of features i and
// i + d/2), two query elements, eight f16 pairs out.
template <int D>
__global__ void __launch_bounds__(1024) mbuild_kernel(PoolGeom g, PlanDev p, int layer,
                                                     const uint16_t* __restrict__ q) {
  using namespace dec;
  constexpr int NF = D / 2;
  // the decode grid may be scheduled now; it waits for this grid's
  // completion before reading M
  asm volatile("griddepcontrol.launch_dependents;");
  const uint8_t* ws = g.base + g.off_ws;
  // the pair's record (its agents' pool ids, ranks, scales and q rows were
  // looked up by the host), staged once per block
  __shared__ __align__(16) MPair smp;
  const int tid = threadIdx.x;
  static_assert(sizeof(MPair) % 4 == 0, "MPair is copied as words");
  if (tid < (int)(sizeof(MPair) / 4))
    ((uint32_t*)&smp)[tid] = ((const uint32_t*)((const MPair*)(ws + p.off_mpairs) + blockIdx.y))[tid];
  __syncthreads();
  const MPair& mp = smp;
  const int* s_pa = mp.pool_agent;
  const int* s_rp = mp.rp;
  const float* s_s = mp.s;
  const int32_t* s_qrow = mp.qrow;
  // one block per pair (few SMs busy, so most decode CTAs start at once);
  // each thread takes units tid, tid + 1024, ...
  const int n_units = (mp.zcols / kRPA / 8) * kRPA * NF;
#pragma unroll 2
  for (int u = tid; u < n_units; u += blockDim.x) {
  const int i = u % NF, gq = (u / NF) % kRPA, j = u / (NF * kRPA);
  // owning agent of rank group j
  int col = 0, ai = 0;
  for (int a = 0; a < mp.n_agents; ++a) {
    if (8 * j >= col && 8 * j < col + s_rp[a]) { ai = a; break; }
    col += s_rp[a];
  }
  const int rp = s_rp[ai], pa = s_pa[ai];
  const float sa = s_s[ai];
  const int64_t qrow = s_qrow[ai * kRPA + gq];
  const __nv_bfloat16* qp = (const __nv_bfloat16*)(q + qrow * D);
  const __nv_bfloat16* bk = (const __nv_bfloat16*)(g.base + g.off_bk + (int64_t)pa * g.bk_agent_bytes) +
                            ((int64_t)layer * g.H_kv + mp.head) * (int64_t)D * g.rmax_pad;
  const int RC = rp / 8, kc = (8 * j - col) / 8, i1 = i + NF;
  const float x0 = sa * __bfloat162float(qp[i]), x1 = sa * __bfloat162float(qp[i1]);
  const uint4 b0 = *(const uint4*)(bk + ((i / 8) * RC + kc) * 64 + (i % 8) * 8);
  const uint4 b1 = *(const uint4*)(bk + ((i1 / 8) * RC + kc) * 64 + (i1 % 8) * 8);
  const uint32_t w0[4] = {b0.x, b0.y, b0.z, b0.w}, w1[4] = {b1.x, b1.y, b1.z, b1.w};
  uint8_t* M = (uint8_t*)ws + mp.mofs;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // column n = (8 j + e) * 4 + gq: group n / 8 = 4 j + e / 2, row n % 8 =
    // 4 (e % 2) + gq; features 2i, 2i + 1
    const float bi = (e & 1) ? bf_hi(w0[e / 2]) : bf_lo(w0[e / 2]);
    const float bh = (e & 1) ? bf_hi(w1[e / 2]) : bf_lo(w1[e / 2]);
    *(uint32_t*)(M + ((4 * j + e / 2) * (D / 8) + i / 4) * 128 + (4 * (e & 1) + gq) * 16 + (i % 4) * 4) =
        pack_h2(x0 * bi + x1 * bh, x1 * bi - x0 * bh);
  }
}
  }

// ============================================================ launcher ==

template <int D, bool COMP>
static int launch_decode_t(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q,
                           cudaStream_t st) {
  using LY = dec::Layout<D, COMP>;
  static_assert(LY::TOTAL <= 232448, "shared memory over the 227 KB a CTA may use");
  static PerDeviceOnce once;
  const int se = once.run([] {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, COMP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL);
    if (e != cudaSuccess) return (int)e;
    // the warps' register split (setmaxnreg) hands out exactly the block's
    // launch registers, 512 x 128: a build with another count would leave
    // the compute warps waiting for registers, so it is refused here
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, decode_kernel<D, COMP>);
    if (e != cudaSuccess) return (int)e;
    return fa.numRegs == 128 ? 0 : (int)cudaErrorInvalidConfiguration;
  });
  if (se != 0) return se;
  mbuild_kernel<D><<<dim3(1, p.n_mpairs), 1024, 0, st>>>(g, p, layer, q);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  // programmatic dependent launch: the decode grid's set-up overlaps the M
  // build; it waits for that grid before its first copy of M
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_ctas);
  cfg.blockDim = dim3(dec::kThreads);
  cfg.dynamicSmemBytes = LY::TOTAL;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, decode_kernel<D, COMP>, g, p, layer, q);
}

bool decode_applies(const PoolGeom& g, const PlanDev& p) {
  return g.G * p.C == dec::kRPA && (g.d == 64 || g.d == 128);
}

int launch_decode(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q,
                  int compressed, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (g.d == 128)
    return compressed ? launch_decode_t<128, true>(g, p, layer, q, st)
                      : launch_decode_t<128, false>(g, p, layer, q, st);
  return compressed ? launch_decode_t<64, true>(g, p, layer, q, st)
                    : launch_decode_t<64, false>(g, p, layer, q, st);
}

}  // namespace fk
