// Residual (low-rank) prefill: Lk = X A_k and Lv = X A_v for a run of a
// forked agent's tokens, written straight into its rCache.
//
// ForkKV guide, "Two-Tier Lookup Mechanics", case B (base cache hit, no
// residual for this adapter: only the low-rank projection X A_i is
// computed) and LRAgent summary, "BaseShared" (the "LR prefill" each agent
// needs over the accumulated context).
//
// One CTA per 128-token tile.  The contraction over d_model runs on the
// tensor cores (tcgen05, kind::f16, bf16 operands, fp32 accumulators in
// TMEM): D[128 tokens x N] with N = 2 rp, columns [0, rp) for A_k and
// [rp, 2 rp) for A_v (rank columns past r are zero).  Operands are staged
// by the CTA's threads into K-major no-swizzle core matrices, 128 features
// of d_model per chunk, two chunks in flight: the loads of a chunk overlap
// the MMAs of the one before.  The epilogue rounds to bf16 (nearest even)
// and writes the rCache layouts (Lk as [T/8][rp/8][8 keys][8 ranks], Lv as
// [T/8][rp/8][8 ranks][8 keys]).  Every wait is bounded; a timeout sets the
// pool's error word and the CTA writes nothing.
#include <cuda_runtime.h>

#include <cstdint>

#include "fk_device.cuh"
#include "fk_internal.h"

namespace fk {
namespace pre {

constexpr int kThreads = 256;
constexpr int kTile = 128;            // tokens per CTA (the MMA's M)
constexpr int kChunk = 128;           // d_model features per pipeline stage
constexpr int kXBytes = kTile * kChunk * 2;

template <int NB>
struct Layout {
  static constexpr int W_B = kChunk * NB * 2;
  static constexpr int STAGE = kXBytes + W_B;
  static constexpr int TOTAL = 2 * STAGE;
};

}  // namespace pre

template <int NB>
__global__ void __launch_bounds__(pre::kThreads, 1)
    lr_prefill_kernel(PoolGeom g, uint8_t* __restrict__ lk_base, uint8_t* __restrict__ lv_base,
                      int r, int rp, int pos, int n, int d_model,
                      const uint16_t* __restrict__ X, const uint16_t* __restrict__ Ak,
                      const uint16_t* __restrict__ Av) {
  using namespace pre;
  using LY = Layout<NB>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[3];   // two stages, final drain
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTile;
  const uint32_t sbase = smem_u32(smem);
  uint32_t* errw = (uint32_t*)(g.base + g.off_err);

  // zero both stages (rank columns past r stay zero), barriers, TMEM
  for (int i = tid * 16; i < LY::TOTAL; i += kThreads * 16) *(uint4*)(smem + i) = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 128);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t idesc = idesc_f16(128, NB, 1);
  uint32_t parb = 0;                  // bit s: parity thread 0 waits for on stage s
  const int n_chunks = d_model / kChunk;

  for (int c = 0; c < n_chunks; ++c) {
    const int s = c & 1;
    uint8_t* xs = smem + s * LY::STAGE;
    uint8_t* wsm = xs + kXBytes;
    // the MMAs of chunk c - 2 read this stage (one thread waits; the CTA
    // leaves the loop together on a timeout)
    if (c >= 2) {
      if (tid == 0) {
        uint32_t ps = (parb >> s) & 1u;
        if (!mbar_wait(smem_u32(&bars[s]), ps, &abort_flag, errw)) abort_flag = 1;
        parb ^= 1u << s;
      }
      __syncthreads();
      if (abort_flag) break;
      tc_fence_after();
    }
    // X: 128 rows x 16 groups of 8 features; (row, group) at group * 2048 + row * 16.
    // A warp takes 8 rows x 4 groups: 64 contiguous bytes of each row from
    // global memory, and 8 distinct 16-byte bank groups per shared store.
#pragma unroll 4
    for (int seg = tid; seg < kTile * (kChunk / 8); seg += kThreads) {
      const int wseg = seg >> 5, ln = seg & 31;
      const int row = (wseg % 16) * 8 + (ln & 7), kg = (wseg / 16) * 4 + (ln >> 3);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t0 + row < n) v = __ldg((const uint4*)(X + (int64_t)(t0 + row) * d_model + c * kChunk + kg * 8));
      *(uint4*)(xs + kg * (kTile * 16) + row * 16) = v;
    }
    // W = [A_k | A_v]: element (column nn, feature k) at (k / 8) * NB * 16 + nn * 16 + (k % 8) * 2
    const int cg = r / 8;                                  // 8-column groups of one of A_k, A_v
#pragma unroll 2
    for (int seg = tid; seg < kChunk * 2 * cg; seg += kThreads) {
      const int k = seg / (2 * cg), which = (seg / cg) % 2, gq = seg % cg;
      const uint16_t* src = (which ? Av : Ak) + (int64_t)(c * kChunk + k) * r + gq * 8;
      const uint4 v = __ldg((const uint4*)src);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      const int nn0 = which * rp + gq * 8;
      uint8_t* dst = wsm + (k / 8) * (NB * 16) + (k % 8) * 2;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *(uint16_t*)(dst + (nn0 + e) * 16) = (uint16_t)((e & 1) ? (w4[e / 2] >> 16) : (w4[e / 2] & 0xFFFFu));
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // thread 0 issues every MMA and commit, so that its final commit below
    // tracks all of them
    if (warp == 0) {
      if (lane == 0 && !abort_flag) {
        const uint64_t dA = sdesc(sbase + s * LY::STAGE, kTile * 16, 128);
        const uint64_t dB = sdesc(sbase + s * LY::STAGE + kXBytes, NB * 16, 128);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          mma_ss(tmem, dA + (uint64_t)((ks * 2 * kTile * 16) >> 4), dB + (uint64_t)((ks * 2 * NB * 16) >> 4),
                 idesc, (c > 0 || ks > 0) ? 1u : 0u);
        mma_commit(smem_u32(&bars[s]));
      }
      __syncwarp();
    }
  }
  // every MMA issued (by thread 0, the elected lane of warp 0) completes
  // before the epilogue reads TMEM or TMEM is freed, also after a timeout
  if (tid == 0) {
    mma_commit(smem_u32(&bars[2]));
    if (!mbar_wait_drain(smem_u32(&bars[2]), 0)) abort_flag = 1;
  }
  __syncthreads();
  tc_fence_after();
  // epilogue: warps 0-3 own TMEM lanes 0-127 = the tile's tokens
  if (warp < 4 && !abort_flag) {
    const int row = warp * 32 + lane, t = pos + t0 + row;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const bool live = t0 + row < n;
    const int RC = rp / 8;
#pragma unroll
    for (int c0 = 0; c0 < NB; c0 += 32) {
      uint32_t v[32];
      tmem_ld32_wait(tmem + c0 + lane_off, v);
      if (live) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          const int nn = c0 + e;                       // 8 columns nn .. nn + 7
          const bool is_v = nn >= rp;
          const int k0 = is_v ? nn - rp : nn;
          if (k0 < rp) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
              w[h] = pack_bf2(__uint_as_float(v[e + 2 * h]), __uint_as_float(v[e + 2 * h + 1]));
            const int ch = k0 / 8;
            if (!is_v) {
              *(uint4*)(lk_base + ((int64_t)(t / 8) * RC + ch) * 128 + (t % 8) * 16) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              uint16_t* vp = (uint16_t*)(lv_base + ((int64_t)(t / 8) * RC + ch) * 128) + (t % 8);
#pragma unroll
              for (int h = 0; h < 8; ++h) vp[h * 8] = (uint16_t)((h & 1) ? (w[h / 2] >> 16) : (w[h / 2] & 0xFFFFu));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

template <int NB>
static int launch_prefill_t(const PoolGeom& g, uint8_t* lk, uint8_t* lv, int r, int rp, int pos,
                            int n, int d_model, const uint16_t* X, const uint16_t* Ak,
                            const uint16_t* Av, cudaStream_t st) {
  using LY = pre::Layout<NB>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(lr_prefill_kernel<NB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, LY::TOTAL);
    if (e != cudaSuccess) return (int)e;
    attr_done = true;
  }
  const int grid = (n + pre::kTile - 1) / pre::kTile;
  lr_prefill_kernel<NB><<<grid, pre::kThreads, LY::TOTAL, st>>>(g, lk, lv, r, rp, pos, n, d_model,
                                                                 X, Ak, Av);
  return (int)cudaGetLastError();
}

int launch_residual_prefill(const PoolGeom& g, int layer, const AgentDev& ag, int r, int pos, int n,
                            int d_model, const uint16_t* X, const uint16_t* Ak, const uint16_t* Av,
                            void* stream) {
  uint8_t* lk = g.base + ag.rc_off + (int64_t)layer * rc_layer_bytes(g, ag.rp);
  uint8_t* lv = lk + (int64_t)g.tcap * ag.rp * 2;
  cudaStream_t st = (cudaStream_t)stream;
  switch (2 * ag.rp) {
    case 32: return launch_prefill_t<32>(g, lk, lv, r, ag.rp, pos, n, d_model, X, Ak, Av, st);
    case 64: return launch_prefill_t<64>(g, lk, lv, r, ag.rp, pos, n, d_model, X, Ak, Av, st);
    case 96: return launch_prefill_t<96>(g, lk, lv, r, ag.rp, pos, n, d_model, X, Ak, Av, st);
    case 128: return launch_prefill_t<128>(g, lk, lv, r, ag.rp, pos, n, d_model, X, Ak, Av, st);
    default: return (int)cudaErrorInvalidValue;
  }
}

}  // namespace fk
