// Internal declarations shared by the host side (fk_host.cpp) and the
// kernels (fk_kernels.cu).  Not part of the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>

#include "forkkv.h"

#if defined(__CUDACC__)
#define FK_HD __host__ __device__
#else
#define FK_HD
#endif

namespace fk {

constexpr int kPage = 16;          // tokens per page
constexpr int kTileTok = 128;      // tokens per attention tile (8 pages)
constexpr int kTilePages = kTileTok / kPage;
constexpr int kMaxRows = 64;       // query rows of one work tile
constexpr int kMaxRankSum = 64;    // sum of padded ranks of one work tile
constexpr int kMaxAgentsPerTile = 4;
constexpr int kMaxRowGroups = 4;   // 16-row query groups the agents of a tile touch
constexpr int kMaxRankPad = 64;
// Decode-shaped calls with d = 128 on an uncompressed pool run in tiles of
// up to eight agent slots (four query rows each): two halves of four slots,
// each half holding at most 64 padded ranks (fk_decode8.cu).
constexpr int kDecodeSlots = 8;
constexpr int kDecodeHalfRank = 64;
constexpr int kMaxDevices = 64;    // devices a process may drive (per-device set-up tables)

FK_HD inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
FK_HD inline int rank_pad(int r) { return (r + 15) / 16 * 16; }

// Per registered agent; mirrored on the device.
struct AgentDev {
  int32_t rp;              // rank rounded up to 16 (0: not registered)
  float s;                 // residual scale alpha / r
  int64_t rc_off;          // byte offset of layer 0's Lk in the carve-out
};

// Geometry and region offsets of a pool, passed to kernels by value.
struct PoolGeom {
  uint8_t* base;           // device carve-out
  int32_t L, H_q, H_kv, d, G, num_pages, max_agents, rmax_pad;
  int32_t tcap;            // rCache tokens per agent (multiple of 128)
  float rope_base;
  int64_t off_kb, off_vb, off_bk, off_bv, off_agents, off_rope, off_err;
  int64_t off_kq, off_vc, off_vn, off_ks, off_kmax, off_meta, off_ws;
  int64_t off_lvmap;       // per pool agent: 128-byte TMA tensor map of its Lv (all layers)
  int64_t off_trig;        // d = 128: [tcap][d/2] f16 pairs (cos, sin)(t theta_i); else -1
  int64_t ws_bytes, meta_bytes;
  int64_t page_bytes;      // bytes of one (page, head) bf16 block: 16*d*2
  int64_t kb_layer_bytes;  // num_pages * H_kv * page_bytes
  int64_t bk_agent_bytes;  // one agent's BkT for all layers
  int64_t bv_agent_bytes;
  int32_t compressed;
};

// rCache bytes of one layer of one agent (Lk + Lv).
FK_HD inline int64_t rc_layer_bytes(const PoolGeom& g, int rp) {
  return 2LL * g.tcap * rp * 2;
}

// ---------------------------------------------------------------- plans --
// Device-side plan, packed in the workspace.  All offsets are in elements
// of the named array, counted from the workspace start.
struct CallAgent {
  int32_t pool_agent;      // pool agent id
  int32_t seq_len;         // keys of this agent
};

struct PlanDev {
  int32_t n_items, n_rows, n_pages, n_tile_agents, A, C, causal;
  int32_t n_out_rows;      // A * C * H_q
  int32_t n_partials;      // partial slots
  int32_t partial_stride;  // floats per partial slot: d + rmax_pad + 4
  int32_t n_ctas;          // persistent CTAs; CTA c runs items cta[c] .. cta[c+1]-1
  int32_t n_mpairs;        // decode-shaped calls: (agent tile, kv head) pairs with an M
  int32_t n_ditems;        // four-agent decode calls: DecItem records (0 otherwise)
  int32_t chunk;           // 1: the items are the chunk kernel's (fk_chunk.cu)
  int32_t slots8;          // 1: eight-slot decode tiles (fk_decode8.cu); tile_agents holds
                           // kDecodeSlots entries per tile (-1: empty slot), rows 4 per slot
                           // (row_agent -1: a padded row)
  int32_t stall_probe;     // failure-detection test: the four-agent decode kernel's key
                           // warp also waits on a barrier nothing completes (set per call)
  int64_t off_items, off_row_agent, off_row_cg, off_pages, off_tile_agents,
          off_call_agents, off_csr_ptr, off_csr_slots, off_partials, off_cta;
  int64_t off_mpairs;      // MPair[n_mpairs]
  int64_t off_ditems;      // DecItem[n_ditems]
};

// One work item of the four-agent decode kernel (fk_decode.cu) with every
// table lookup done by the host, so that the kernel starts an item with a
// single read.  Records 0 .. n_ctas - 1 are the CTAs' first items (a CTA
// without work has n_pages = 0); `next` chains a CTA's further items
// (-1: none).
struct DecItem {
  int32_t head, n_rows, n_pages, lp_begin, n_ag, partial_begin, page_begin, sum_rp;
  int32_t lv_rp;           // ranks of the Lv^T stage (agents reading the same rows share one block)
  int32_t next;
  int32_t lim_min[2];      // per half of the rows (8 rows): fewest keys any of them sees (0: padded row)
  int32_t rp[kMaxAgentsPerTile], col[kMaxAgentsPerTile], pool_agent[kMaxAgentsPerTile];
  int32_t lvcol[kMaxAgentsPerTile];   // first rank of the agent's block in the Lv^T stage
  float s[kMaxAgentsPerTile];
  int64_t rc_off[kMaxAgentsPerTile];
  int32_t qrow[4 * kMaxAgentsPerTile];     // q row of each query row (-1: padded row)
  int32_t row_lim[4 * kMaxAgentsPerTile];  // keys each query row sees (0: padded row)
  int32_t first_pages[kTilePages];         // page ids of the item's first 128-key tile
  int64_t mofs;            // the item's M (see MPair): byte offset from the workspace start
  int32_t mbytes;
  int32_t split;           // 1: the agents' rows all sit in the first half (at most two
                           // agents) and their rank groups are shared by both halves
};
static_assert(sizeof(DecItem) % 16 == 0, "DecItem is read in 16-byte words");

// One (agent tile, kv head) of a four-agent decode call: the rows of its
// agents and where its query-side RoPE matrix M (d x 4 sum-of-ranks f16, in
// the decode kernel's shared-memory image) sits in the workspace.  The
// host looks up each agent's pool id, padded rank and residual scale and
// each query row's q row, so that building M needs no chain of table loads.
struct MPair {
  int32_t head, agent_begin, n_agents, row_begin;
  int32_t zcols, pad;      // columns of M (4 x the tile's padded rank sum)
  int64_t mofs;            // byte offset from the workspace start
  int32_t pool_agent[kMaxAgentsPerTile], rp[kMaxAgentsPerTile];
  float s[kMaxAgentsPerTile];
  int32_t qrow[kMaxAgentsPerTile * 4];
};

// Host launchers (fk_kernels.cu).  All return a cudaError_t as int.
int launch_base_append(const PoolGeom& g, int layer, const int32_t* page_of_chunk,
                       int n_chunks, int pos, int n, const uint16_t* Kb,
                       const uint16_t* Vb, void* stream);
int launch_residual_append(const PoolGeom& g, int layer, const AgentDev& ag,
                           int r, int pos, int n, const uint16_t* Lk,
                           const uint16_t* Lv, void* stream);
// Lk = X A_k and Lv = X A_v of tokens pos..pos+n-1 on the tensor cores,
// written into the agent's rCache (fk_prefill.cu).  x_map: 128-byte TMA
// tensor map of X ([n][d_model] bf16, 64 x 128 boxes, 128-byte swizzle).
int launch_residual_prefill(const PoolGeom& g, int layer, const AgentDev& ag, int r, int pos,
                            int n, int d_model, const void* x_map, const uint16_t* Ak,
                            const uint16_t* Av, void* stream);
int launch_agent_register(const PoolGeom& g, int agent, int r, int rp,
                          const AgentDev& ag, const uint16_t* Bk,
                          const uint16_t* Bv, void* stream);
int launch_compress(const PoolGeom& g, int layer, const int32_t* d_pages,
                    const int32_t* d_fill, int n_pages, void* stream);
int launch_load_compressed(const PoolGeom& g, int layer, const int32_t* d_pages,
                           int n_pages, const int8_t* kq, const uint8_t* vcodes,
                           const float* vnorm, float k_scale, void* stream);
int launch_attention(const PoolGeom& g, const PlanDev& p, int layer,
                     const uint16_t* q, uint16_t* out, int compressed,
                     int num_sms, void* stream, int* n_launches,
                     void* event_after_main);

// Decode-shaped calls (four query rows per agent: G * C == 4) run the
// decode kernel (fk_decode.cu); the combine is shared.
bool decode_applies(const PoolGeom& g, const PlanDev& p);
int launch_decode(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q,
                  int compressed, void* stream);

// Fills the pool's RoPE table of [cos, sin](t theta_i) for t < tcap (d = 128)
// on the legacy default stream (fk_decode8.cu).
int launch_trig_table(const PoolGeom& g);

// Decode-shaped calls planned in eight-slot tiles (d = 128, uncompressed
// pool) run the eight-agent decode kernel (fk_decode8.cu); the combine is
// shared.
bool decode8_applies(const PoolGeom& g, const PlanDev& p);
int launch_decode8(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q, void* stream);

// Calls with at least 128 query rows per agent and kv head (d = 128,
// uncompressed pool) run the chunk kernel (fk_chunk.cu); the combine is
// shared.
bool chunk_applies(const PoolGeom& g, const PlanDev& p);
int launch_chunk(const PoolGeom& g, const PlanDev& p, int layer, const uint16_t* q, void* stream);

// Device address and size of the static scratch array that
// fk_residual_attention_noalloc uses (looked up once per device).
int noalloc_scratch(void** ptr, size_t* bytes);

}  // namespace fk
