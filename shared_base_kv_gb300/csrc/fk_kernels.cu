// Kernels of libforkkv for sm_103a (GB300).
//
//  * base / residual appends into the pool's tensor-core-native layouts;
//  * agent registration (B matrices laid out for the MMA);
//  * the compressed pool codec (int8 keys, 3-bit FWHT + Lloyd-Max values);
//  * the residual attention kernel (warp-specialised, tcgen05 + TMEM, bulk
//    copies into shared memory) and its split-K combine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fk_device.cuh"
#include "fk_internal.h"
#include "fk_once.h"

namespace fk {

__device__ __forceinline__ uint32_t* err_word(const PoolGeom& g) {
  return (uint32_t*)(g.base + g.off_err);
}
__device__ __forceinline__ void flag_bounds(const PoolGeom& g, uint32_t bit) {
  atomicOr(err_word(g), bit);
}

// ============================================================= appends ==

struct PageList {
  int32_t id[64];
};

// Tokens t in [pos, pos+n) are written; rows of the touched pages past
// pos+n are zeroed (a page is only ever appended to at its end).  One
// thread per (token slot, head, 8-element chunk of d).
__global__ void base_append_kernel(PoolGeom g, int layer, PageList pages, int lp0, int pos, int n,
                                   const uint4* __restrict__ Kb, const uint4* __restrict__ Vb) {
  const int D = g.d, H = g.H_kv, CH = D / 8;
  const int end = ((pos + n + kPage - 1) / kPage) * kPage;
  const int64_t total = (int64_t)(end - pos) * H * CH;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    int ch = (int)(u % CH);
    int h = (int)((u / CH) % H);
    int t = pos + (int)(u / ((int64_t)CH * H));
    int lp = t / kPage, row = t % kPage;
    int32_t page = pages.id[lp - lp0];
    if (page < 0 || page >= g.num_pages) { flag_bounds(g, 1u); continue; }
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (t < pos + n) {
      int64_t src = ((int64_t)(t - pos) * H + h) * CH + ch;
      kv = Kb[src];
      vv = Vb[src];
    }
    int64_t blk = (int64_t)layer * g.kb_layer_bytes + ((int64_t)page * H + h) * g.page_bytes;
    // keys: [token-group][d-chunk][token][8 d]
    uint8_t* kp = g.base + g.off_kb + blk + (((row / 8) * CH + ch) * 128 + (row % 8) * 16);
    *(uint4*)kp = kv;
    // values: [token-chunk][d-group][d][8 tokens]
    uint16_t* vp = (uint16_t*)(g.base + g.off_vb + blk + ((row / 8) * CH + ch) * 128) + (row % 8);
    const uint16_t* ve = (const uint16_t*)&vv;
#pragma unroll
    for (int e = 0; e < 8; ++e) vp[e * 8] = ve[e];
  }
}

// Residual rows: Lk as [token-group][r-chunk][token][8 r], Lv as
// [token-chunk][r-group][r][8 tokens]; padding columns r..rp stay zero.
__global__ void residual_append_kernel(PoolGeom g, uint8_t* lk_base, uint8_t* lv_base, int r,
                                       int rp, int pos, int n, const uint16_t* __restrict__ Lk,
                                       const uint16_t* __restrict__ Lv) {
  const int RC = rp / 8;
  const int64_t total = (int64_t)n * RC;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    int ch = (int)(u % RC);
    int t = pos + (int)(u / RC);
    uint16_t kv[8], vv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      int c = ch * 8 + e;
      kv[e] = c < r ? Lk[(int64_t)(t - pos) * r + c] : (uint16_t)0;
      vv[e] = c < r ? Lv[(int64_t)(t - pos) * r + c] : (uint16_t)0;
    }
    uint8_t* kp = lk_base + ((int64_t)(t / 8) * RC + ch) * 128 + (t % 8) * 16;
    *(uint4*)kp = *(uint4*)kv;
    uint16_t* vp = (uint16_t*)(lv_base + ((int64_t)(t / 8) * RC + ch) * 128) + (t % 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) vp[e * 8] = vv[e];
  }
}

// B matrices: BkT per (layer, head) as [d-group][r-chunk][d][8 r] (the MMA
// operand of Lk Bk), Bv row-major [layer][rmax_pad][H_kv*d]; rows past the
// rank are zero.
__global__ void agent_register_kernel(PoolGeom g, int agent, int r, int rp,
                                      const uint16_t* __restrict__ Bk,
                                      const uint16_t* __restrict__ Bv) {
  const int D = g.d, H = g.H_kv, HD = H * D, RC = rp / 8;
  const int64_t total = (int64_t)g.L * g.rmax_pad * HD;
  uint16_t* bkt = (uint16_t*)(g.base + g.off_bk + (int64_t)agent * g.bk_agent_bytes);
  uint16_t* bv = (uint16_t*)(g.base + g.off_bv + (int64_t)agent * g.bv_agent_bytes);
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    int col = (int)(u % HD);
    int k = (int)((u / HD) % g.rmax_pad);
    int l = (int)(u / ((int64_t)HD * g.rmax_pad));
    uint16_t bkv = 0, bvv = 0;
    if (k < r) {
      int64_t src = ((int64_t)l * r + k) * HD + col;
      bkv = Bk[src];
      bvv = Bv[src];
    }
    bv[((int64_t)l * g.rmax_pad + k) * HD + col] = bvv;
    if (k < rp) {
      int h = col / D, dd = col % D;
      int64_t blk = ((int64_t)l * H + h) * (int64_t)D * g.rmax_pad;
      bkt[blk + ((dd / 8) * RC + k / 8) * 64 + (dd % 8) * 8 + (k % 8)] = bkv;
    }
  }
}

// ============================================================ codec =====


__device__ __forceinline__ float bf16_at(const uint8_t* p) {
  return __bfloat162float(*(const __nv_bfloat16*)p);
}

// Address of key element (row, dd) of a (layer, page, head) block.
__device__ __forceinline__ const uint8_t* key_at(const PoolGeom& g, int layer, int page, int h,
                                                 int row, int dd) {
  const int CH = g.d / 8;
  int64_t blk = (int64_t)layer * g.kb_layer_bytes + ((int64_t)page * g.H_kv + h) * g.page_bytes;
  return g.base + g.off_kb + blk + ((row / 8) * CH + dd / 8) * 128 + (row % 8) * 16 + (dd % 8) * 2;
}
__device__ __forceinline__ const uint8_t* val_at(const PoolGeom& g, int layer, int page, int h,
                                                 int row, int dd) {
  const int CH = g.d / 8;
  int64_t blk = (int64_t)layer * g.kb_layer_bytes + ((int64_t)page * g.H_kv + h) * g.page_bytes;
  return g.base + g.off_vb + blk + ((row / 8) * CH + dd / 8) * 128 + (dd % 8) * 16 + (row % 8) * 2;
}

// max |K| over the live rows of the listed pages (float bits of |x| order
// like unsigned integers).
__global__ void kmax_kernel(PoolGeom g, int layer, const int32_t* __restrict__ pages,
                            const int32_t* __restrict__ fill, int n_pages) {
  const int D = g.d, H = g.H_kv;
  float m = 0.f;
  const int64_t total = (int64_t)n_pages * kPage * H * D;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    int dd = (int)(u % D);
    int h = (int)((u / D) % H);
    int row = (int)((u / ((int64_t)D * H)) % kPage);
    int pi = (int)(u / ((int64_t)D * H * kPage));
    if (row >= fill[pi]) continue;
    m = fmaxf(m, fabsf(bf16_at(key_at(g, layer, pages[pi], h, row, dd))));
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax((unsigned int*)(g.base + g.off_kmax) + layer, __float_as_uint(m));
}

// One warp per (page, row, head): int8 keys with the layer scale, and the
// value vector's norm and 3-bit codes of z = H v / n.
__global__ void encode_kernel(PoolGeom g, int layer, const int32_t* __restrict__ pages,
                              const int32_t* __restrict__ fill, int n_pages) {
  const int D = g.d, H = g.H_kv, PER = D / 32, NB = D / 8;
  const int lane = threadIdx.x & 31;
  const float kmax = __uint_as_float(((const unsigned int*)(g.base + g.off_kmax))[layer]);
  const float scale = kmax > 0.f ? __fdiv_rn(kmax, 127.f) : 1.f;
  if (blockIdx.x == 0 && threadIdx.x == 0) ((float*)(g.base + g.off_ks))[layer] = scale;
  const int64_t units = (int64_t)n_pages * kPage * H;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; w < units;
       w += (int64_t)gridDim.x * blockDim.x / 32) {
    int h = (int)(w % H);
    int row = (int)((w / H) % kPage);
    int pi = (int)(w / ((int64_t)H * kPage));
    int page = pages[pi];
    int64_t tok = (((int64_t)layer * g.num_pages + page) * H + h) * kPage + row;
    // tokens are laid out [L][num_pages][H][16]; keys [..][d], codes [..][3d/8]
    int8_t* kq = (int8_t*)(g.base + g.off_kq) + tok * D;
    uint8_t* vc = g.base + g.off_vc + tok * (3 * D / 8);
    float* vn = (float*)(g.base + g.off_vn) + tok;
    bool live = row < fill[pi];
    float v[4];
    for (int e = 0; e < PER; ++e) {
      int dd = lane * PER + e;
      float k = live ? bf16_at(key_at(g, layer, page, h, row, dd)) : 0.f;
      float qv = fminf(fmaxf(rintf(__fdiv_rn(k, scale)), -127.f), 127.f);
      kq[dd] = (int8_t)qv;
      v[e] = live ? bf16_at(val_at(g, layer, page, h, row, dd)) : 0.f;
    }
    float ss = 0.f;
    for (int e = 0; e < PER; ++e) ss = fmaf(v[e], v[e], ss);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    float nrm = sqrtf(ss);
    // unnormalised FWHT, natural order: in-thread stages, then across lanes
    for (int hh = 1; hh < PER; hh <<= 1)
      for (int e = 0; e < PER; ++e)
        if (!(e & hh)) { float a = v[e], b = v[e + hh]; v[e] = a + b; v[e + hh] = a - b; }
    for (int hl = 1; hl < 32; hl <<= 1) {
      for (int e = 0; e < PER; ++e) {
        float o = __shfl_xor_sync(0xffffffffu, v[e], hl);
        v[e] = (lane & hl) ? (o - v[e]) : (v[e] + o);
      }
    }
    uint32_t code[4];
    for (int e = 0; e < PER; ++e) {
      float z = nrm > 0.f ? __fdiv_rn(v[e], nrm) : 0.f;
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < 7; ++j) c += (z >= 0.5f * (c_lloyd[j] + c_lloyd[j + 1])) ? 1u : 0u;
      code[e] = c;
    }
    // bit planes: plane b, code i at bit i%8 of byte i/8
    for (int b = 0; b < 3; ++b) {
      uint32_t bits = 0;
      for (int e = 0; e < PER; ++e) bits |= ((code[e] >> b) & 1u) << e;   // PER bits of this lane
      // byte j collects codes 8j..8j+7 = lanes (8j/PER) .. ; gather via shuffles
      uint32_t byte = 0;
      const int lanes_per_byte = 8 / PER;
      for (int q = 0; q < lanes_per_byte; ++q) {
        uint32_t other = __shfl_sync(0xffffffffu, bits, (lane / lanes_per_byte) * lanes_per_byte + q);
        byte |= other << (q * PER);
      }
      if (lane % lanes_per_byte == 0) vc[b * NB + lane / lanes_per_byte] = (uint8_t)byte;
    }
    if (lane == 0) *vn = live ? nrm : 0.f;
  }
}

__global__ void load_compressed_kernel(PoolGeom g, int layer, const int32_t* __restrict__ pages,
                                       int n_pages, const int8_t* __restrict__ kq,
                                       const uint8_t* __restrict__ vc,
                                       const float* __restrict__ vn, float k_scale) {
  const int D = g.d, H = g.H_kv, VB = 3 * D / 8;
  if (blockIdx.x == 0 && threadIdx.x == 0) ((float*)(g.base + g.off_ks))[layer] = k_scale;
  const int64_t units = (int64_t)n_pages * kPage * H;   // (page, row, head)
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units;
       u += (int64_t)gridDim.x * blockDim.x) {
    int h = (int)(u % H);
    int row = (int)((u / H) % kPage);
    int pi = (int)(u / ((int64_t)H * kPage));
    int page = pages[pi];
    if (page < 0 || page >= g.num_pages) { flag_bounds(g, 4u); continue; }
    int64_t dst = (((int64_t)layer * g.num_pages + page) * H + h) * kPage + row;
    int64_t src = ((int64_t)pi * kPage + row) * H + h;
    for (int e = 0; e < D; e += 16)
      *(uint4*)((int8_t*)(g.base + g.off_kq) + dst * D + e) = *(const uint4*)(kq + src * D + e);
    for (int e = 0; e < VB; e += 16)
      *(uint4*)(g.base + g.off_vc + dst * VB + e) = *(const uint4*)(vc + src * VB + e);
    ((float*)(g.base + g.off_vn))[dst] = vn[src];
  }
}

// ========================================================= attention =====
//
// One persistent CTA per SM walks the work items.  Each item is one kv head,
// up to 64 query rows of up to 4 agents (sum of padded ranks <= 64) that
// name the same physical pages over a run of logical pages.  The run is cut
// into 128-token tiles; per tile:
//   producer warp : bulk-copies the tile's Kb pages, each agent's Lk rows,
//                   and (one tile ahead) the Vb pages and Lv rows to smem;
//   MMA warp      : S  = Kb Q^T                     (TMEM, tokens x rows)
//                   U_a = Lk_a Bk_a^T  per agent    (TMEM, tokens x d, fp32)
//                   S += R_a (Q s_a)^T per agent    (A operand from TMEM)
//                   O^T += Vb^T P^T, OL_a += P Lv_a, L += P 1
//   compute WG    : R_a = RoPE_t(U_a) in f16, written back over U_a; masked
//                   online softmax of S (rescaling O, OL, L only when a
//                   row's running max grows by more than 2^8); P in bf16.
// Per item the compute warpgroup writes the split partial (m, l, O, OL)
// of every row; the combine kernel merges splits and applies Bv once.

namespace attn {

constexpr int kThreads = 384;
constexpr int kPRowGroup = 2304;        // P: 16 token-chunks x 144 B
constexpr int kPChunk = 144;
constexpr int kA = kMaxAgentsPerTile;
// TMEM columns
constexpr uint32_t kTmS = 0, kTmU0 = 64, kTmU1 = 192, kTmOT = 320, kTmOL = 384;
constexpr int kOnesLane = 64;   // lane of OL^T that sums P (row sums)
// Lv^T stage: per token-chunk 9 r-groups (8 of ranks, 1 of ones).  The M=128
// MMA reads 16 r-groups; groups 9..15 fall in the next chunk (finite data,
// lanes 72..127 of OL^T are never used).
constexpr int kLvChunk = 9 * 128;

template <int D, bool COMP>
struct Layout {
  static constexpr int PAGE_B = kPage * D * 2;
  static constexpr int P_B = 8 * kPRowGroup;
  static constexpr int KB_B = kTilePages * PAGE_B;
  static constexpr int LK_B = kMaxRankSum * kTileTok * 2;
  static constexpr int VB_B = KB_B;
  static constexpr int LV_B = 16 * kLvChunk;    // Lv^T of all agents + ones row, per token-chunk
  static constexpr int BK_B = kMaxRankSum * D * 2;
  static constexpr int Q_B = kMaxRows * D * 2;
  static constexpr int QM_B = 4 * 16 * D * 2;
  static constexpr int ONES_B = 0;
  static constexpr int KQ_B = COMP ? kTilePages * kPage * D : 0;
  static constexpr int VC_B = COMP ? kTilePages * kPage * (3 * D / 8) : 0;
  static constexpr int VN_B = COMP ? kTilePages * kPage * 4 : 0;
  static constexpr int oP = 0;
  static constexpr int oKB = oP + P_B;              // the OL MMA reads 16 row-groups of P:
  static constexpr int oLK0 = oKB + KB_B;           // the 8 past P_B fall in KB/LK (finite)
  static constexpr int oLK1 = COMP ? oLK0 : oLK0 + LK_B;   // one Lk buffer when compressed
  static constexpr int oVB = oLK1 + LK_B;
  static constexpr int oLV = oVB + VB_B;            // d=64 reads 1 KB past VB: lands in LV
  static constexpr int oBK = oLV + LV_B;
  static constexpr int oQ = oBK + BK_B;
  static constexpr int oQM = oQ + Q_B;
  static constexpr int oONES = oQM + QM_B;
  static constexpr int oKQ = oONES + ONES_B;
  static constexpr int oVC = oKQ + KQ_B;
  static constexpr int oVN = oVC + VC_B;
  static constexpr int TAU_B = (D / 2) * 128 * 4;      // per-thread tau rotations, [word][lane]
  static constexpr int oTAU = (oVN + VN_B + 127) / 128 * 128;
  static constexpr int oMISC = oTAU + TAU_B;
  static constexpr int MISC_B = 4096;
  static constexpr int TOTAL = oMISC + MISC_B;
};

// barrier indices
enum {
  B_KB_FULL, B_KB_EMPTY, B_LK_FULL0, B_LK_FULL1, B_LK_EMPTY0, B_LK_EMPTY1, B_VL_FULL,
  B_VL_EMPTY, B_BK_FULL, B_BK_EMPTY, B_Q_FULL, B_Q_EMPTY, B_U_FULL0, B_U_FULL1, B_R_FULL0,
  B_R_FULL1, B_UFREE0, B_UFREE1, B_S_FULL, B_S_EMPTY, B_P_FULL, B_PV_DONE, B_ACC_EMPTY,
  B_KQ_FULL, B_KQ_EMPTY, B_VC_FULL, B_VC_EMPTY, B_FINAL, B_ROT_FULL0, B_ROT_FULL1,
  B_ROT_EMPTY0, B_ROT_EMPTY1, B_COUNT
};
// Arrival counts: 1 = one thread or an MMA commit, 4 = one lane per warp of
// a warpgroup, 2 = the value stage of the compressed pool (the producer's
// transaction count plus the dequantiser).
__host__ __device__ constexpr uint32_t bar_count(int i, bool comp) {
  return (i == B_Q_FULL || i == B_R_FULL0 || i == B_R_FULL1 || i == B_S_EMPTY || i == B_P_FULL ||
          i == B_ACC_EMPTY || i == B_ROT_EMPTY0 || i == B_ROT_EMPTY1)
             ? 4u
             : (i == B_VL_FULL && comp) ? 2u : 1u;
}
// barriers a role waits on as "empty" start one phase ahead
constexpr uint32_t kEmptyMask = (1u << B_KB_EMPTY) | (1u << B_LK_EMPTY0) | (1u << B_LK_EMPTY1) |
                                (1u << B_VL_EMPTY) | (1u << B_BK_EMPTY) | (1u << B_Q_EMPTY) |
                                (1u << B_UFREE0) | (1u << B_UFREE1) | (1u << B_S_EMPTY) |
                                (1u << B_ACC_EMPTY) | (1u << B_KQ_EMPTY) | (1u << B_VC_EMPTY) |
                                (1u << B_ROT_EMPTY0) | (1u << B_ROT_EMPTY1);

struct Misc {
  uint64_t bar[B_COUNT];
  uint32_t tmem_base;
  int abort_flag;
  float m_used[kMaxRows];
  float alpha[kMaxRows];
  float red[4][kMaxRows];
  int32_t row_T[kMaxRows];
  int32_t row_pos[kMaxRows];
  uint32_t rot[2][64];           // tile-start rotations, a 2-tile ring: f16x2 cos pairs, sin pairs
  float theta[64];               // RoPE theta_i
  unsigned long long frac[64];   // theta_i / (2 pi) as a 64-bit binary fraction
};

static_assert(sizeof(Misc) <= 4096, "Misc must fit its smem slot (Layout::MISC_B)");

// What every role derives from a work item.  Per-agent arrays are only
// indexed with compile-time indices (unrolled loops), so they stay in
// registers.
struct ItemInfo {
  int head, n_rows, nrp, n_pages, lp_begin, n_ag, partial_begin, row_begin, n_tiles, page_begin;
  int rp[kA], col[kA], g0[kA], ng[kA], ra0[kA], ra1[kA], call_agent[kA], pool_agent[kA], qm[kA];
  float s[kA];
  int64_t rc_off[kA];
};

__device__ __forceinline__ void load_item(const PoolGeom& g, const PlanDev& p, const uint8_t* ws,
                                          int it, ItemInfo& I) {
  const fk_work_item& w = ((const fk_work_item*)(ws + p.off_items))[it];
  const int32_t* tile_agents = (const int32_t*)(ws + p.off_tile_agents);
  const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
  const AgentDev* ag = (const AgentDev*)(g.base + g.off_agents);
  I.head = w.head;
  I.n_rows = w.n_rows;
  I.nrp = (w.n_rows + 15) / 16 * 16;
  I.n_pages = w.n_pages;
  I.lp_begin = w.lp_begin;
  I.n_ag = w.n_agents;
  I.partial_begin = w.partial_begin;
  I.row_begin = w.row_begin;
  I.page_begin = w.page_begin;
  I.n_tiles = (w.n_pages + kTilePages - 1) / kTilePages;
  const int rpa = g.G * p.C;
  int col = 0, qm = 0;
#pragma unroll
  for (int a = 0; a < kA; ++a) {
    I.rp[a] = 0; I.ng[a] = 0; I.g0[a] = 0; I.col[a] = col; I.qm[a] = qm; I.s[a] = 0.f;
    I.rc_off[a] = 0; I.call_agent[a] = -1; I.pool_agent[a] = 0; I.ra0[a] = 0; I.ra1[a] = 0;
    if (a < I.n_ag) {
      int ci = tile_agents[w.agent_begin + a];
      int pa = ca[ci].pool_agent;
      AgentDev dv = ag[pa];
      I.call_agent[a] = ci;
      I.pool_agent[a] = pa;
      I.rp[a] = dv.rp;
      I.s[a] = dv.s;
      I.rc_off[a] = dv.rc_off;
      col += dv.rp;
      if (I.n_ag == 1) { I.ra0[a] = 0; I.ra1[a] = w.n_rows; }
      else { I.ra0[a] = a * rpa; I.ra1[a] = (a + 1) * rpa; }
      I.g0[a] = I.ra0[a] / 16;
      I.ng[a] = (I.ra1[a] - 1) / 16 - I.g0[a] + 1;
      qm += I.ng[a];
    }
  }
}

__device__ __forceinline__ const uint8_t* rc_lk(const PoolGeom& g, const ItemInfo& I, int a,
                                                int layer) {
  return g.base + I.rc_off[a] + (int64_t)layer * rc_layer_bytes(g, I.rp[a]);
}
__device__ __forceinline__ const uint8_t* rc_lv(const PoolGeom& g, const ItemInfo& I, int a,
                                                int layer) {
  return rc_lk(g, I, a, layer) + (int64_t)g.tcap * I.rp[a] * 2;
}

}  // namespace attn

// Masked online softmax of one tile for NRP (16/32/48/64) padded query
// rows, run by the softmax warpgroup (lane = token): scores from TMEM, the
// running max of a row moves only when the row's tile max exceeds it by more
// than 2^8 (then O^T and OL^T are rescaled in TMEM), P in bf16 to smem in the
// K-major layout of the PV MMAs.  Rows past n_rows have row_T = 0 and come
// out as P = 0.
template <int NRP, int D, bool COMP, typename Wait>
__device__ __forceinline__ void softmax_tile(uint8_t* smem, attn::Misc& M, uint32_t tmem,
                                             uint32_t lane_off, int ln, int sw, int lane, int k,
                                             int t0, int ntok, int n_rows, float scale_log2,
                                             Wait& wait, uint32_t bar_s_empty) {
  using namespace attn;
  using LY = Layout<D, COMP>;
  wait(B_S_FULL);
  tc_fence_after();
  uint32_t sv[NRP];                 // scores, then log2-domain scores (float bits)
#pragma unroll
  for (int c0 = 0; c0 < NRP; c0 += 16) tmem_ld16(tmem + kTmS + c0 + lane_off, sv + c0);
  tmem_wait_ld();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_s_empty);
  const int tabs = t0 + ln;
  bool need = false;
#pragma unroll
  for (int j = 0; j < NRP; ++j) {
    bool ok = ln < ntok && tabs < M.row_T[j] && tabs <= M.row_pos[j];
    float s = ok ? __uint_as_float(sv[j]) * scale_log2 : -INFINITY;
    sv[j] = __float_as_uint(s);
    need |= s > M.m_used[j] + 8.f;
  }
  int any;
  asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 3, 128, p; selp.u32 %0, 1, 0, q; }"
               : "=r"(any) : "r"((int)need));
  if (k > 0) wait(B_PV_DONE);
  if (any) {
#pragma unroll
    for (int j = 0; j < NRP; ++j) {
      float v = __uint_as_float(sv[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) M.red[sw][j] = v;
    }
    named_bar(2, 128);
    if (ln < NRP) {
      float al = 1.f;
      if (ln < n_rows) {
        float cm = fmaxf(fmaxf(M.red[0][ln], M.red[1][ln]), fmaxf(M.red[2][ln], M.red[3][ln]));
        float mo = M.m_used[ln];
        float mn = fmaxf(mo, cm);
        if (mn > mo) { al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn); M.m_used[ln] = mn; }
      }
      M.alpha[ln] = al;
    }
    named_bar(2, 128);
    if (k > 0) {
      tc_fence_after();
      uint32_t raw[16];
#pragma unroll
      for (int c0 = 0; c0 < NRP; c0 += 16) {
        tmem_ld16(tmem + kTmOT + c0 + lane_off, raw);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[c0 + e]);
        tmem_st16(tmem + kTmOT + c0 + lane_off, raw);
        tmem_ld16(tmem + kTmOL + c0 + lane_off, raw);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) raw[e] = __float_as_uint(__uint_as_float(raw[e]) * M.alpha[c0 + e]);
        tmem_st16(tmem + kTmOL + c0 + lane_off, raw);
      }
      tmem_wait_st();
    }
  }
  const int tc = ln / 8, tr = ln % 8;
#pragma unroll
  for (int j = 0; j < NRP; ++j) {
    float m = M.m_used[j];
    float s = __uint_as_float(sv[j]);
    float pv = (s == -INFINITY || m == -INFINITY) ? 0.f : exp2f(s - m);
    *(__nv_bfloat16*)(smem + LY::oP + (j / 8) * kPRowGroup + tc * kPChunk + (j % 8) * 16 + tr * 2) =
        __float2bfloat16_rn(pv);
  }
}

template <int D, bool COMP>
__global__ void __launch_bounds__(attn::kThreads, 1)
    attention_kernel(PoolGeom g, PlanDev p, int layer, const uint16_t* __restrict__ q) {
  using namespace attn;
  using LY = Layout<D, COMP>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc& M = *reinterpret_cast<Misc*>(smem + LY::oMISC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* ws = g.base + g.off_ws;
  const int32_t* cta_items = (const int32_t*)(ws + p.off_cta);
  uint32_t* errw = err_word(g);
  volatile int* abort_flag = &M.abort_flag;
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return smem_u32(&M.bar[i]); };
  // Each role keeps the parity it waits for on barrier i in bit i.
  uint32_t ph = kEmptyMask;
  auto wait = [&](int i) {
    uint32_t par = (ph >> i) & 1u;
    const bool ok = mbar_wait(bar(i), par, abort_flag, errw);
    ph ^= 1u << i;
    return ok;
  };
  // the producer posts a transaction count and copies only after a wait
  // that succeeded while the CTA carries on: after a given-up wait the
  // stage's previous phase may still be pending
  auto go = [&](int i) { return wait(i) && !*abort_flag; };
  // the dependent combine grid may be scheduled now; it waits for this
  // grid's completion before reading the partials
  asm volatile("griddepcontrol.launch_dependents;");

  // ---- set-up: zero smem (junk rows read by padded MMAs stay finite),
  // ones row of the Lv^T stage, RoPE tables, barriers, TMEM.
  for (int i = tid * 16; i < LY::TOTAL; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int i = tid; i < 16 * 8; i += kThreads)
    ((uint16_t*)(smem + LY::oLV + (i / 8) * kLvChunk + (kOnesLane / 8) * 128))[i % 8] = 0x3F80;
  if (tid < 64) {
    M.theta[tid] = ((const float*)(g.base + g.off_rope))[tid];
    M.frac[tid] = ((const unsigned long long*)(g.base + g.off_rope + 256))[tid];
  }
  __syncthreads();
  if (tid >= 128 && tid < 256) {
    // rotation by each tile offset tau = tid - 128 (f16 pairs), kept in smem
    // as [word][lane] so that a warp reads 32 consecutive words
    const int tau = tid - 128;
    uint32_t* T = (uint32_t*)(smem + LY::oTAU);
    for (int j = 0; j < D / 4; ++j) {
      float c0, s0, c1, s1;
      sincosf((float)tau * M.theta[2 * j], &s0, &c0);
      sincosf((float)tau * M.theta[2 * j + 1], &s1, &c1);
      T[j * 128 + tau] = pack_h2(c0, c1);
      T[(D / 4 + j) * 128 + tau] = pack_h2(s0, s1);
    }
  }
  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), bar_count(i, COMP));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&M.tmem_base), 512);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_base;

  if (warp == 0 && lane == 0) {
    // ================================================== producer ====
    int tile_ctr = 0;
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      const int32_t* pages = (const int32_t*)(ws + p.off_pages) + I.page_begin;
      if (go(B_BK_EMPTY)) {
        uint32_t bytes = 0;
#pragma unroll
        for (int a = 0; a < kA; ++a) bytes += D * I.rp[a] * 2;
        mbar_expect_tx(bar(B_BK_FULL), bytes);
#pragma unroll
        for (int a = 0; a < kA; ++a)
          if (a < I.n_ag) {
            const uint8_t* src = g.base + g.off_bk + (int64_t)I.pool_agent[a] * g.bk_agent_bytes +
                                 ((int64_t)layer * g.H_kv + I.head) * (int64_t)D * g.rmax_pad * 2;
            bulk_g2s(sbase + LY::oBK + I.col[a] * D * 2, src, D * I.rp[a] * 2, bar(B_BK_FULL));
          }
      }
      // keys of tile k, then the values of tile k-1 (consumed one tile later)
      auto load_values = [&](int k) {
        const int p0 = k * kTilePages;
        const int np = min(kTilePages, I.n_pages - p0);
        const int t0 = (I.lp_begin + p0) * kPage;
        if (COMP && go(B_VC_EMPTY)) {
          mbar_expect_tx(bar(B_VC_FULL), np * kPage * (3 * D / 8 + 4));
          for (int j = 0; j < np; ++j) {
            int pg = pages[p0 + j];
            int64_t tok = (((int64_t)layer * g.num_pages + pg) * g.H_kv + I.head) * kPage;
            bulk_g2s(sbase + LY::oVC + j * kPage * (3 * D / 8), g.base + g.off_vc + tok * (3 * D / 8),
                     kPage * (3 * D / 8), bar(B_VC_FULL));
            bulk_g2s(sbase + LY::oVN + j * kPage * 4, g.base + g.off_vn + tok * 4, kPage * 4,
                     bar(B_VC_FULL));
          }
        }
        if (!go(B_VL_EMPTY)) return;
        const int ntok = min(kTileTok, g.tcap - t0);
        uint32_t bytes = COMP ? 0 : np * LY::PAGE_B;
#pragma unroll
        for (int a = 0; a < kA; ++a) bytes += ntok * I.rp[a] * 2;
        mbar_expect_tx(bar(B_VL_FULL), bytes);
        if (!COMP)
          for (int j = 0; j < np; ++j) {
            int pg = pages[p0 + j];
            const uint8_t* src = g.base + g.off_vb + (int64_t)layer * g.kb_layer_bytes +
                                 ((int64_t)pg * g.H_kv + I.head) * LY::PAGE_B;
            bulk_g2s(sbase + LY::oVB + j * LY::PAGE_B, src, LY::PAGE_B, bar(B_VL_FULL));
          }
#pragma unroll
        for (int a = 0; a < kA; ++a)
          if (a < I.n_ag) {
            const uint8_t* src = rc_lv(g, I, a, layer) + (int64_t)t0 * I.rp[a] * 2;
            const int cb = I.rp[a] * 16;            // one token-chunk of this agent
            for (int c = 0; c < ntok / 8; ++c)
              bulk_g2s(sbase + LY::oLV + c * kLvChunk + (I.col[a] / 8) * 128, src + c * cb, cb,
                       bar(B_VL_FULL));
          }
      };
      for (int k = 0; k < I.n_tiles; ++k, ++tile_ctr) {
        const int p0 = k * kTilePages;
        const int np = min(kTilePages, I.n_pages - p0);
        const int t0 = (I.lp_begin + p0) * kPage;
        if (!COMP) {
          if (go(B_KB_EMPTY)) {
          mbar_expect_tx(bar(B_KB_FULL), np * LY::PAGE_B);
          for (int j = 0; j < np; ++j) {
            int pg = pages[p0 + j];
            const uint8_t* src = g.base + g.off_kb + (int64_t)layer * g.kb_layer_bytes +
                                 ((int64_t)pg * g.H_kv + I.head) * LY::PAGE_B;
            bulk_g2s(sbase + LY::oKB + j * LY::PAGE_B, src, LY::PAGE_B, bar(B_KB_FULL));
          }
          }
        } else if (go(B_KQ_EMPTY)) {
          mbar_expect_tx(bar(B_KQ_FULL), np * kPage * D);
          for (int j = 0; j < np; ++j) {
            int pg = pages[p0 + j];
            const uint8_t* src = g.base + g.off_kq +
                                 ((((int64_t)layer * g.num_pages + pg) * g.H_kv + I.head) * kPage) * D;
            bulk_g2s(sbase + LY::oKQ + j * kPage * D, src, kPage * D, bar(B_KQ_FULL));
          }
        }
        {
          const int b = COMP ? 0 : (tile_ctr & 1);
          if (go(B_LK_EMPTY0 + b)) {
          const int ntok = min(kTileTok, g.tcap - t0);
          uint32_t bytes = 0;
#pragma unroll
          for (int a = 0; a < kA; ++a) bytes += ntok * I.rp[a] * 2;
          mbar_expect_tx(bar(B_LK_FULL0 + b), bytes);
#pragma unroll
          for (int a = 0; a < kA; ++a)
            if (a < I.n_ag)
              bulk_g2s(sbase + (b ? LY::oLK1 : LY::oLK0) + I.col[a] * kTileTok * 2,
                       rc_lk(g, I, a, layer) + (int64_t)t0 * I.rp[a] * 2, ntok * I.rp[a] * 2,
                       bar(B_LK_FULL0 + b));
          }
        }
        if (k > 0) load_values(k - 1);
      }
      load_values(I.n_tiles - 1);
    }
  } else if (warp == 1 && lane == 0) {
    // ===================================================== MMA issuer ====
    int tile_ctr = 0;
    const uint32_t t_S = tmem + kTmS, t_OT = tmem + kTmOT, t_OL = tmem + kTmOL;
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      wait(B_BK_FULL);
      wait(B_Q_FULL);
      tc_fence_after();
      const uint32_t id_S = idesc_f16(128, I.nrp, 1);
      const uint32_t id_U = idesc_f16(128, D, 1);
      const uint32_t id_PV = idesc_f16(128, I.nrp, 1);
      auto residual = [&](int a) {   // a: compile-time after unrolling
        const int b = a & 1;
        wait(B_R_FULL0 + b);
        tc_fence_after();
        const uint32_t id_R = idesc_f16(128, 16 * I.ng[a], 0);
        const uint32_t t_R = tmem + (b ? kTmU1 : kTmU0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ts(t_S + 16 * I.g0[a], t_R + 8 * ks,
                 sdesc(sbase + LY::oQM + I.qm[a] * 16 * D * 2 + ks * 128, (D / 16) * 128, (D / 8) * 128),
                 id_R, 1);
        mma_commit(bar(B_UFREE0 + b));
      };
      auto pv = [&](int j) {
        wait(B_P_FULL);
        wait(B_VL_FULL);
        if (j == 0) wait(B_ACC_EMPTY);
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < kTileTok / 16; ++ks) {
          const uint32_t acc = (j == 0 && ks == 0) ? 0u : 1u;
          const uint64_t dP = sdesc(sbase + LY::oP + ks * 2 * kPChunk, kPChunk, kPRowGroup);
          mma_ss(t_OT, sdesc(sbase + LY::oVB + ks * LY::PAGE_B, (D / 8) * 128, 128), dP, id_PV, acc);
          mma_ss(t_OL, sdesc(sbase + LY::oLV + ks * 2 * kLvChunk, kLvChunk, 128), dP, id_PV, acc);
        }
        mma_commit(bar(B_VL_EMPTY));
        mma_commit(bar(B_PV_DONE));
      };
      for (int k = 0; k < I.n_tiles; ++k, ++tile_ctr) {
        wait(B_S_EMPTY);
        wait(B_KB_FULL);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(t_S, sdesc(sbase + LY::oKB + ks * 256, 128, (D / 8) * 128),
                 sdesc(sbase + LY::oQ + ks * 256, 128, (D / 8) * 128), id_S, ks > 0 ? 1u : 0u);
        mma_commit(bar(B_KB_EMPTY));
        const int lb = COMP ? 0 : (tile_ctr & 1);
        wait(B_LK_FULL0 + lb);
        tc_fence_after();
        const uint32_t lk_base = sbase + (lb ? LY::oLK1 : LY::oLK0);
#pragma unroll
        for (int a = 0; a < kA; ++a) {
          if (a < I.n_ag) {
            const int b = a & 1;
            wait(B_UFREE0 + b);
            tc_fence_after();
            const int rc = I.rp[a] / 8;
            const uint32_t t_U = tmem + (b ? kTmU1 : kTmU0);
            for (int ks = 0; ks < I.rp[a] / 16; ++ks)
              mma_ss(t_U, sdesc(lk_base + I.col[a] * kTileTok * 2 + ks * 256, 128, rc * 128),
                     sdesc(sbase + LY::oBK + I.col[a] * D * 2 + ks * 256, 128, rc * 128), id_U,
                     ks > 0 ? 1u : 0u);
            mma_commit(bar(B_U_FULL0 + b));
            if (a > 0) residual(a - 1);
          }
        }
        mma_commit(bar(B_LK_EMPTY0 + lb));
#pragma unroll
        for (int a = 0; a < kA; ++a)
          if (a == I.n_ag - 1) residual(a);
        mma_commit(bar(B_S_FULL));
        if (k > 0) pv(k - 1);
      }
      pv(I.n_tiles - 1);
      mma_commit(bar(B_Q_EMPTY));
      mma_commit(bar(B_BK_EMPTY));
    }
    // every MMA issued completes before tensor memory is freed, also after
    // a given-up wait (the drain ignores the abort flag)
    mma_commit(bar(B_FINAL));
    mbar_wait_drain(bar(B_FINAL), (ph >> B_FINAL) & 1u);
  } else if (warp == 2) {
    // =========================== tile-start rotations, one tile ahead ====
    // Exact t0 * theta_i reduced modulo 2 pi with a 64-bit binary fraction,
    // then an accurate sincos; lane j writes the f16 pairs of freqs 2j, 2j+1.
    int tile_ctr = 0;
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      for (int k = 0; k < I.n_tiles; ++k, ++tile_ctr) {
        const int b = tile_ctr & 1;
        wait(B_ROT_EMPTY0 + b);
        const int t0 = (I.lp_begin + k * kTilePages) * kPage;
        if (lane < D / 4) {
          float cc[2], ssn[2];
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            unsigned long long fr = (unsigned long long)t0 * M.frac[2 * lane + z];
            float ang = (float)(unsigned int)(fr >> 32) * 1.4629180792671596e-09f;  // 2 pi / 2^32
            if (ang > 3.14159265f) ang -= 6.28318531f;
            sincosf(ang, &ssn[z], &cc[z]);
          }
          M.rot[b][lane] = pack_h2(cc[0], cc[1]);
          M.rot[b][32 + lane] = pack_h2(ssn[0], ssn[1]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ROT_FULL0 + b));
      }
    }
  } else if (COMP && warp == 3) {
    // ====================================== dequantiser (compressed pool) ====
    const float kscale = ((const float*)(g.base + g.off_ks))[layer];
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      for (int k = 0; k < I.n_tiles; ++k) {
        const int np = min(kTilePages, I.n_pages - k * kTilePages);
        // keys: int8 [page][16][D] -> bf16 (value * scale) in the key layout
        wait(B_KQ_FULL);
        wait(B_KB_EMPTY);
        for (int u = lane; u < np * kPage * (D / 8); u += 32) {
          int ch = u % (D / 8), row = (u / (D / 8)) % kPage, pj = u / (kPage * (D / 8));
          const int8_t* src = (const int8_t*)(smem + LY::oKQ) + (pj * kPage + row) * D + ch * 8;
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf2((float)src[2 * e] * kscale, (float)src[2 * e + 1] * kscale);
          *(uint4*)(smem + LY::oKB + pj * LY::PAGE_B + ((row / 8) * (D / 8) + ch) * 128 + (row % 8) * 16) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) { mbar_arrive(bar(B_KB_FULL)); mbar_arrive(bar(B_KQ_EMPTY)); }
        // values: codes -> level * n / D in the value layout (rotated domain)
        wait(B_VC_FULL);
        wait(B_VL_EMPTY);
        for (int u = lane; u < np * 2 * (D / 8); u += 32) {
          int dg = u % (D / 8), tc = (u / (D / 8)) % 2, pj = u / (2 * (D / 8));
          float w8[8];
          uint32_t c8[8];
#pragma unroll
          for (int tt = 0; tt < 8; ++tt) {
            int row = tc * 8 + tt;
            const uint8_t* cb = smem + LY::oVC + (pj * kPage + row) * (3 * D / 8);
            uint32_t b0 = cb[dg], b1 = cb[D / 8 + dg], b2 = cb[2 * (D / 8) + dg];
            c8[tt] = b0 | (b1 << 8) | (b2 << 16);
            w8[tt] = ((const float*)(smem + LY::oVN))[pj * kPage + row] * (1.0f / D);
          }
          uint8_t* dst = smem + LY::oVB + pj * LY::PAGE_B + (tc * (D / 8) + dg) * 128;
#pragma unroll
          for (int e = 0; e < 8; ++e) {   // d = 8 dg + e
            uint32_t w[4];
#pragma unroll
            for (int h2 = 0; h2 < 4; ++h2) {
              float v2[2];
#pragma unroll
              for (int z = 0; z < 2; ++z) {
                uint32_t cc = c8[2 * h2 + z];
                uint32_t code = ((cc >> e) & 1u) | (((cc >> (8 + e)) & 1u) << 1) | (((cc >> (16 + e)) & 1u) << 2);
                v2[z] = c_lloyd[code] * w8[2 * h2 + z];
              }
              w[h2] = pack_bf2(v2[0], v2[1]);
            }
            *(uint4*)(dst + e * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) { mbar_arrive(bar(B_VL_FULL)); mbar_arrive(bar(B_VC_EMPTY)); }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ================================================ RoPE warpgroup ====
    const int ln = tid - 128;                          // TMEM lane = token
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t* TAU = (const uint32_t*)(smem + LY::oTAU);
    int tile_ctr = 0;
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      const int n_ag = I.n_ag;
      for (int k = 0; k < I.n_tiles; ++k, ++tile_ctr) {
        // rotation of this thread's token: tile start (ring) composed with
        // its offset in the tile
        const int rb = tile_ctr & 1;
        wait(B_ROT_FULL0 + rb);
        uint32_t Cp[D / 4], Sp[D / 4];
#pragma unroll
        for (int j = 0; j < D / 4; ++j) {
          __half2 c0 = as_h2(M.rot[rb][j]), s0 = as_h2(M.rot[rb][32 + j]);
          __half2 ct = as_h2(TAU[j * 128 + ln]), st = as_h2(TAU[(D / 4 + j) * 128 + ln]);
          Cp[j] = as_u32(__hfma2(c0, ct, __hneg2(__hmul2(s0, st))));
          Sp[j] = as_u32(__hfma2(s0, ct, __hmul2(c0, st)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_ROT_EMPTY0 + rb));
        // RoPE of each agent's residual keys, written back as f16 pairs
        for (int a = 0; a < n_ag; ++a) {
          const int b = a & 1;
          const uint32_t t_U = tmem + (b ? kTmU1 : kTmU0) + lane_off;
          wait(B_U_FULL0 + b);
          tc_fence_after();
#pragma unroll
          for (int cb = 0; cb < D / 16; cb += 4) {
            uint32_t lo[4][8], hi[4][8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              tmem_ld8(t_U + 8 * (cb + c), lo[c]);
              tmem_ld8(t_U + D / 2 + 8 * (cb + c), hi[c]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int ci = cb + c;
              uint32_t r8[8];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                __half2 xl = __floats2half2_rn(__uint_as_float(lo[c][2 * j]), __uint_as_float(lo[c][2 * j + 1]));
                __half2 xh = __floats2half2_rn(__uint_as_float(hi[c][2 * j]), __uint_as_float(hi[c][2 * j + 1]));
                __half2 C = as_h2(Cp[4 * ci + j]), S = as_h2(Sp[4 * ci + j]);
                r8[j] = as_u32(__hfma2(xl, C, __hneg2(__hmul2(xh, S))));
                r8[4 + j] = as_u32(__hfma2(xh, C, __hmul2(xl, S)));
              }
              tmem_st8(t_U + 8 * ci, r8);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_R_FULL0 + b));
        }
      }
    }
  } else if (warp >= 8) {
    // ============================================= softmax warpgroup ====
    const int ln = tid - 256;                          // TMEM lane = token / d / row
    const int sw = warp - 8;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float scale_log2 = 1.4426950408889634f * rsqrtf((float)D);
    for (int it = cta_items[blockIdx.x]; it < cta_items[blockIdx.x + 1]; ++it) {
      ItemInfo I;
      load_item(g, p, ws, it, I);
      const int n_rows = I.n_rows, nrp = I.nrp, n_ag = I.n_ag;
      const int32_t* row_agent = (const int32_t*)(ws + p.off_row_agent) + I.row_begin;
      const int32_t* row_cg = (const int32_t*)(ws + p.off_row_cg) + I.row_begin;
      const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
      // ---- stage Q (bf16) and per-agent s_a * Q (f16, other agents' rows 0)
      wait(B_Q_EMPTY);
      if (ln < kMaxRows) {
        M.m_used[ln] = -INFINITY;
        M.row_T[ln] = 0;
        M.row_pos[ln] = -1;
        if (ln < n_rows) {
          int ci = row_agent[ln];
          int T = ca[ci].seq_len;
          int c = row_cg[ln] / g.G;
          M.row_T[ln] = T;
          M.row_pos[ln] = p.causal ? (T - p.C + c) : 0x7fffffff;
        }
      }
      for (int u = ln; u < nrp * (D / 8); u += 128) {
        int row = u / (D / 8), ch = u % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < n_rows) {
          int ci = row_agent[row], cg = row_cg[row];
          int c = cg / g.G, gg = cg % g.G;
          int64_t qrow = ((int64_t)ci * p.C + c) * g.H_q + I.head * g.G + gg;
          v = *(const uint4*)(q + qrow * D + ch * 8);
        }
        *(uint4*)(smem + LY::oQ + ((row / 8) * (D / 8) + ch) * 128 + (row % 8) * 16) = v;
      }
#pragma unroll
      for (int a = 0; a < kA; ++a) {
        if (a < n_ag) {
          for (int u = ln; u < I.ng[a] * 16 * (D / 8); u += 128) {
            int lr = u / (D / 8), ch = u % (D / 8);
            int row = I.g0[a] * 16 + lr;
            uint32_t w[4] = {0, 0, 0, 0};
            if (row >= I.ra0[a] && row < I.ra1[a] && row < n_rows) {
              int ci = row_agent[row], cg = row_cg[row];
              int c = cg / g.G, gg = cg % g.G;
              int64_t qrow = ((int64_t)ci * p.C + c) * g.H_q + I.head * g.G + gg;
              const __nv_bfloat16* src = (const __nv_bfloat16*)(q + qrow * D + ch * 8);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_h2(__bfloat162float(src[2 * e]) * I.s[a], __bfloat162float(src[2 * e + 1]) * I.s[a]);
            }
            *(uint4*)(smem + LY::oQM + I.qm[a] * 16 * D * 2 + ((lr / 8) * (D / 8) + ch) * 128 + (lr % 8) * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_proxy_async();
      named_bar(2, 128);                 // row tables visible to every softmax warp
      if (lane == 0) mbar_arrive(bar(B_Q_FULL));

      for (int k = 0; k < I.n_tiles; ++k) {
        const int t0 = (I.lp_begin + k * kTilePages) * kPage;
        const int ntok = min(kTileTok, (I.n_pages - k * kTilePages) * kPage);
        switch (nrp) {
          case 16: softmax_tile<16, D, COMP>(smem, M, tmem, lane_off, ln, sw, lane, k, t0, ntok, n_rows, scale_log2, wait, bar(B_S_EMPTY)); break;
          case 32: softmax_tile<32, D, COMP>(smem, M, tmem, lane_off, ln, sw, lane, k, t0, ntok, n_rows, scale_log2, wait, bar(B_S_EMPTY)); break;
          case 48: softmax_tile<48, D, COMP>(smem, M, tmem, lane_off, ln, sw, lane, k, t0, ntok, n_rows, scale_log2, wait, bar(B_S_EMPTY)); break;
          default: softmax_tile<64, D, COMP>(smem, M, tmem, lane_off, ln, sw, lane, k, t0, ntok, n_rows, scale_log2, wait, bar(B_S_EMPTY)); break;
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL));
      }
      // ---- epilogue: write this item's split partials
      wait(B_PV_DONE);
      tc_fence_after();
      float* part = (float*)(ws + p.off_partials);
      const int PS = p.partial_stride;
      {
        uint32_t raw[16];
        for (int c0 = 0; c0 < nrp; c0 += 16) {
          tmem_ld16(tmem + kTmOT + c0 + lane_off, raw);
          tmem_wait_ld();
          if (ln < D) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c0 + e < n_rows) part[(int64_t)(I.partial_begin + c0 + e) * PS + 4 + ln] = __uint_as_float(raw[e]);
          }
        }
        // OL^T lane ln: residual column r = ln - col of the agent whose
        // columns hold ln (rows of that agent take it), or the row sums.
        int oa = -1, orr = 0;
#pragma unroll
        for (int a = 0; a < kA; ++a)
          if (a < n_ag && ln >= I.col[a] && ln < I.col[a] + I.rp[a]) { oa = a; orr = ln - I.col[a]; }
        int ra0 = 0, ra1 = 0;
#pragma unroll
        for (int a = 0; a < kA; ++a)
          if (a == oa) { ra0 = I.ra0[a]; ra1 = I.ra1[a]; }
        for (int c0 = 0; c0 < nrp; c0 += 16) {
          tmem_ld16(tmem + kTmOL + c0 + lane_off, raw);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = c0 + e;
            if (j < n_rows) {
              float* dst = part + (int64_t)(I.partial_begin + j) * PS;
              if (ln == kOnesLane) dst[1] = __uint_as_float(raw[e]);
              if (oa >= 0 && j >= ra0 && j < ra1) dst[4 + D + orr] = __uint_as_float(raw[e]);
            }
          }
        }
        if (ln < n_rows) part[(int64_t)(I.partial_begin + ln) * PS] = M.m_used[ln];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY));
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

// ============================================================ combine ====
// One CTA of D threads per output row: merge the row's split partials
// (log-sum-exp in base 2), apply Bv once to the merged P Lv (LRAgent
// summary, section 3), rotate the value sum of a compressed pool back
// (inverse FWHT), normalise, round to bf16.
constexpr int kCombineSlotCache = 512;   // split slots of a row staged in shared memory

template <int D, bool COMP>
__global__ void __launch_bounds__(4 * D) combine_kernel(PoolGeom g, PlanDev p, int layer,
                                                        uint16_t* __restrict__ out) {
  __shared__ float sol[kMaxRankPad];
  __shared__ float sx[D];
  __shared__ float qo[4][D], qol[4][kMaxRankPad], qm[4], ql[4];
  __shared__ uint16_t sbv[kMaxRankPad * D];         // this row's Bv slice, [rank][D]
  __shared__ int32_t sslot[kCombineSlotCache];
  const int row = blockIdx.x, d = threadIdx.x % D, qq = threadIdx.x / D;
  const uint8_t* ws = g.base + g.off_ws;
  const int32_t* ptr = (const int32_t*)(ws + p.off_csr_ptr);
  const int32_t* slots = (const int32_t*)(ws + p.off_csr_slots);
  const float* part = (const float*)(ws + p.off_partials);
  const CallAgent* ca = (const CallAgent*)(ws + p.off_call_agents);
  const AgentDev* ag = (const AgentDev*)(g.base + g.off_agents);
  const int PS = p.partial_stride;
  const int hq = row % g.H_q;
  const int i = row / (g.H_q * p.C);
  const int h = hq / g.G;
  const int pa = ca[i].pool_agent;
  const AgentDev dv = ag[pa];
  const int b = ptr[row], e = ptr[row + 1];
  // The plan tables, the agent table and Bv were written before the
  // attention grid started: stage this row's slots and Bv slice while that
  // grid is still running (the launch is programmatic), so that only the
  // partials are read after the wait.
  {
    const uint16_t* bvb = (const uint16_t*)(g.base + g.off_bv + (int64_t)pa * g.bv_agent_bytes) +
                          (int64_t)layer * g.rmax_pad * g.H_kv * D + h * D;
    for (int idx = threadIdx.x; idx < dv.rp * D; idx += 4 * D)
      sbv[idx] = bvb[(int64_t)(idx / D) * g.H_kv * D + idx % D];
    const int ns = min(e - b, kCombineSlotCache);
    for (int j = threadIdx.x; j < ns; j += 4 * D) sslot[j] = slots[b + j];
  }
  __syncthreads();
  auto slot = [&](int k) { return k - b < kCombineSlotCache ? sslot[k - b] : slots[k]; };
  // partials are written by the preceding attention grid
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // four thread groups take every fourth split (a log-sum-exp merge with a
  // running maximum each, all their loads issued first), then group 0
  // merges the four
  const bool has_r = d < dv.rp;
  float Mx = -INFINITY, L = 0.f, o = 0.f, ol = 0.f;
  auto merge = [&](float m, float l, float ov, float olv) {
    if (m == -INFINITY) return;                // a split that saw no visible key
    const float nm = fmaxf(Mx, m);
    const float a = (Mx == -INFINITY) ? 0.f : exp2f(Mx - nm);
    const float w = exp2f(m - nm);
    L = L * a + w * l;
    o = o * a + w * ov;
    ol = ol * a + w * olv;
    Mx = nm;
  };
  int k = b + qq;
  for (; k + 12 < e; k += 16) {
    float m[4], l[4], ov[4], olv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* s = part + (int64_t)slot(k + 4 * j) * PS;
      m[j] = s[0];
      l[j] = s[1];
      ov[j] = s[4 + d];
      olv[j] = has_r ? s[4 + D + d] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) merge(m[j], l[j], ov[j], olv[j]);
  }
  for (; k < e; k += 4) {
    const float* s = part + (int64_t)slot(k) * PS;
    merge(s[0], s[1], s[4 + d], has_r ? s[4 + D + d] : 0.f);
  }
  qo[qq][d] = o;
  if (d < kMaxRankPad) qol[qq][d] = ol;
  if (d == 0) { qm[qq] = Mx; ql[qq] = L; }
  __syncthreads();
  if (qq != 0) return;
  Mx = -INFINITY; L = 0.f; o = 0.f; ol = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) merge(qm[j], ql[j], qo[j][d], d < kMaxRankPad ? qol[j][d] : 0.f);
  if (d < kMaxRankPad) sol[d] = d < dv.rp ? ol : 0.f;
  if (COMP) {
    sx[d] = o;
    asm volatile("bar.sync 1, %0;" ::"r"(D) : "memory");
    for (int hh = 1; hh < D; hh <<= 1) {      // unnormalised FWHT, natural order
      const float a0 = sx[d & ~hh], a1 = sx[d | hh];
      asm volatile("bar.sync 1, %0;" ::"r"(D) : "memory");
      sx[d] = (d & hh) ? (a0 - a1) : (a0 + a1);
      asm volatile("bar.sync 1, %0;" ::"r"(D) : "memory");
    }
    o = sx[d];
  } else {
    asm volatile("bar.sync 1, %0;" ::"r"(D) : "memory");
  }
  // up-projection of the merged low-rank value sum: (sum_t p_t Lv_t) Bv
  float up = 0.f;
#pragma unroll 8
  for (int kk = 0; kk < dv.rp; ++kk) {
    const uint16_t u = sbv[kk * D + d];
    up = fmaf(sol[kk], __bfloat162float(*(const __nv_bfloat16*)&u), up);
  }
  __nv_bfloat16 r = __float2bfloat16_rn((o + dv.s * up) / L);
  out[(int64_t)row * D + d] = *(uint16_t*)&r;
}

// ============================================================ launchers ==

static int grid_for(int64_t work, int per_block) {
  int64_t b = (work + per_block - 1) / per_block;
  return (int)(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}



int launch_base_append(const PoolGeom& g, int layer, const int32_t* page_of_chunk, int n_chunks,
                       int pos, int n, const uint16_t* Kb, const uint16_t* Vb, void* stream) {
  PageList pl;
  for (int i = 0; i < 64; ++i) pl.id[i] = i < n_chunks ? page_of_chunk[i] : -1;
  int lp0 = pos / kPage;
  int end = ((pos + n + kPage - 1) / kPage) * kPage;
  int64_t work = (int64_t)(end - pos) * g.H_kv * (g.d / 8);
  base_append_kernel<<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(
      g, layer, pl, lp0, pos, n, (const uint4*)Kb, (const uint4*)Vb);
  return (int)cudaGetLastError();
}

int launch_residual_append(const PoolGeom& g, int layer, const AgentDev& ag, int r, int pos, int n,
                           const uint16_t* Lk, const uint16_t* Lv, void* stream) {
  uint8_t* lk = g.base + ag.rc_off + (int64_t)layer * rc_layer_bytes(g, ag.rp);
  uint8_t* lv = lk + (int64_t)g.tcap * ag.rp * 2;
  int64_t work = (int64_t)n * (ag.rp / 8);
  residual_append_kernel<<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(g, lk, lv, r, ag.rp,
                                                                                 pos, n, Lk, Lv);
  return (int)cudaGetLastError();
}

int launch_agent_register(const PoolGeom& g, int agent, int r, int rp, const AgentDev&,
                          const uint16_t* Bk, const uint16_t* Bv, void* stream) {
  int64_t work = (int64_t)g.L * g.rmax_pad * g.H_kv * g.d;
  agent_register_kernel<<<grid_for(work, 256), 256, 0, (cudaStream_t)stream>>>(g, agent, r, rp, Bk, Bv);
  return (int)cudaGetLastError();
}

int launch_compress(const PoolGeom& g, int layer, const int32_t* d_pages, const int32_t* d_fill,
                    int n_pages, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(g.base + g.off_kmax + 4LL * layer, 0, 4, st);
  if (e != cudaSuccess) return (int)e;
  if (n_pages > 0) {
    int64_t work = (int64_t)n_pages * kPage * g.H_kv * g.d;
    kmax_kernel<<<grid_for(work, 256 * 8), 256, 0, st>>>(g, layer, d_pages, d_fill, n_pages);
    int64_t units = (int64_t)n_pages * kPage * g.H_kv;
    encode_kernel<<<grid_for(units * 32, 256), 256, 0, st>>>(g, layer, d_pages, d_fill, n_pages);
  } else {
    encode_kernel<<<1, 32, 0, st>>>(g, layer, d_pages, d_fill, 0);
  }
  return (int)cudaGetLastError();
}

int launch_load_compressed(const PoolGeom& g, int layer, const int32_t* d_pages, int n_pages,
                           const int8_t* kq, const uint8_t* vc, const float* vn, float k_scale,
                           void* stream) {
  int64_t units = (int64_t)n_pages * kPage * g.H_kv;
  load_compressed_kernel<<<grid_for(units, 256), 256, 0, (cudaStream_t)stream>>>(
      g, layer, d_pages, n_pages, kq, vc, vn, k_scale);
  return (int)cudaGetLastError();
}

template <int D, bool COMP>
static int launch_attn_t(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q,
                         uint16_t* out, int num_sms, cudaStream_t st, cudaEvent_t ev) {
  using LY = attn::Layout<D, COMP>;
  static PerDeviceOnce once;
  const int se = once.run([] {
    return (int)cudaFuncSetAttribute(attention_kernel<D, COMP>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL);
  });
  if (se != 0) return se;
  if (p.chunk) {
    if (COMP || !chunk_applies(g, p)) return (int)cudaErrorInvalidValue;   // planner mismatch
    int ce = launch_chunk(g, p, layer, q, st);
    if (ce != 0) return ce;
  } else if (p.slots8) {
    if (COMP || !decode8_applies(g, p)) return (int)cudaErrorInvalidValue;  // planner mismatch
    int de = launch_decode8(g, p, layer, q, st);
    if (de != 0) return de;
  } else if (decode_applies(g, p)) {
    int de = launch_decode(g, p, layer, q, COMP ? 1 : 0, st);
    if (de != 0) return de;
  } else {
    attention_kernel<D, COMP><<<p.n_ctas, attn::kThreads, LY::TOTAL, st>>>(g, p, layer, q);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  if (ev) {
    e = cudaEventRecord(ev, st);
    if (e != cudaSuccess) return (int)e;
  }
  // the combine may be launched while the attention grid drains; it waits
  // for that grid inside (programmatic dependent launch)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.n_out_rows);
  cfg.blockDim = dim3(4 * D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, combine_kernel<D, COMP>, g, p, layer, out);
  return (int)e;
}

int launch_attention(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q,
                     uint16_t* out, int compressed, int num_sms, void* stream, int* n_launches,
                     void* event_after_main) {
  cudaStream_t st = (cudaStream_t)stream;
  cudaEvent_t ev = (cudaEvent_t)event_after_main;
  *n_launches = (!p.slots8 && !p.chunk && decode_applies(g, p)) ? 3 : 2;   // (M build,) attention, combine
  if (g.d == 128) {
    return compressed ? launch_attn_t<128, true>(g, p, layer, q, out, num_sms, st, ev)
                      : launch_attn_t<128, false>(g, p, layer, q, out, num_sms, st, ev);
  }
  return compressed ? launch_attn_t<64, true>(g, p, layer, q, out, num_sms, st, ev)
                    : launch_attn_t<64, false>(g, p, layer, q, out, num_sms, st, ev);
}

// Scratch of fk_residual_attention_noalloc (work list and split partials of
// one call), so that the call needs no allocation.  Host code must not pass
// this symbol to a kernel: its host-side name is only a stand-in; the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FK_NOALLOC_SCRATCH_BYTES];

int noalloc_scratch(void** ptr, size_t* bytes) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return (int)e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  *bytes = FK_NOALLOC_SCRATCH_BYTES;
  return 0;
}


}  // namespace fk
