// Residual (low-rank) prefill: Lk = X A_k and Lv = X A_v for a run of a
// forked agent's tokens, written straight into its rCache.
//
// ForkKV guide, "Two-Tier Lookup Mechanics", case B (base cache hit, no
// residual for this adapter: only the low-rank projection X A_i is
// computed) and LRAgent summary, "BaseShared" (the "LR prefill" each agent
// needs over the accumulated context).
//
// One CTA per 128-token tile; the contraction over d_model runs on the
// tensor cores (tcgen05, kind::f16, bf16 operands, fp32 accumulators in
// TMEM): D[128 tokens x N] with N = 2 rp, columns [0, rp) for A_k and
// [rp, 2 rp) for A_v (rank columns past r are zero).  The work streams X,
// so the kernel is a pipeline over chunks of 128 features of d_model, S
// stages deep:
//   warp 0     loads a chunk: X by TMA as two 128-row x 64-feature boxes
//              with the 128-byte swizzle the MMA reads directly (rows past
//              n come back as zeros), and the chunk's 128 rows of A_k and
//              A_v, contiguous in memory, by bulk copy;
//   warps 2-5  transpose the A rows ([k][r] as stored) into the K-major
//              core matrices of the MMA's B operand with ldmatrix.trans
//              (each store fills one whole 128-byte core matrix), then, at
//              the end, read the accumulators back and write the rCache
//              layouts (Lk as [T/8][rp/8][8 keys][8 ranks], Lv as
//              [T/8][rp/8][8 ranks][8 keys], bf16 nearest even);
//   warp 1     allocates TMEM and issues the MMAs of a chunk once its X has
//              landed and its B operand is written.
// Every wait is bounded; a timeout sets the pool's error word, the CTA
// writes nothing, and copies and MMAs still in flight are waited for before
// the CTA releases its shared and tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "fk_device.cuh"
#include "fk_internal.h"
#include "fk_once.h"

namespace fk {
namespace pre {

constexpr int kThreads = 192;
constexpr int kTile = 128;            // tokens per CTA (the MMA's M)
constexpr int kChunk = 128;           // d_model features per pipeline stage
constexpr int kBox = 64;              // features per X box (128 bytes: one swizzle row)
constexpr int kXBytes = kTile * kChunk * 2;

template <int R>
struct Layout {
  static constexpr int RP = (R + 15) / 16 * 16;   // padded rank
  static constexpr int NB = 2 * RP;               // MMA N: [A_k | A_v]
  // [A_k | A_v] chunk as K-major core matrices; the chunk's rows of A_k and
  // A_v land here as stored ([128][r] each) and are transposed in place
  static constexpr int W_B = kChunk * NB * 2;
  static constexpr int STAGE = kXBytes + W_B;      // a multiple of 1024
  static constexpr int S0 = (227 * 1024 - 2048) / STAGE;
  static constexpr int S = S0 > 6 ? 6 : S0;
  static constexpr int BYTES = S * STAGE + 1024;            // + slack for 1024-byte alignment
};

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle:
// 8-row groups 1024 bytes apart; the leading offset is not used.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// OR of `pred` over the 128 threads of warps 2-5 (named barrier 2), the
// same result in every one of them.
__device__ __forceinline__ bool bar_any(bool pred) {
  uint32_t res;
  asm volatile(
      "{ .reg .pred q, p; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 2, 128, q; selp.u32 %0, 1, 0, p; }"
      : "=r"(res)
      : "r"((uint32_t)pred)
      : "memory");
  return res != 0;
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* v) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr)
               : "memory");
}

}  // namespace pre

// R: the agent's rank (a multiple of 8, at most 64), a compile-time
// constant so that the transposer's block indexing folds away.
template <int R>
__global__ void __launch_bounds__(pre::kThreads, 1)
    lr_prefill_kernel(const __grid_constant__ CUtensorMap xmap, PoolGeom g,
                      uint8_t* __restrict__ lk_base, uint8_t* __restrict__ lv_base, int pos,
                      int n, int d_model, const uint16_t* __restrict__ Ak,
                      const uint16_t* __restrict__ Av) {
  using namespace pre;
  using LY = Layout<R>;
  constexpr int S = LY::S, RP = LY::RP, NB = LY::NB, r = R;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[3 * S + 1];   // full, empty, B ready per stage; done
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kTile;
  const uint32_t sraw = smem_u32(smem_raw);
  const uint32_t sbase = (sraw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - sraw);
  uint32_t* errw = (uint32_t*)(g.base + g.off_err);
  auto FULL = [&](int s) { return smem_u32(&bars[s]); };
  auto EMPTY = [&](int s) { return smem_u32(&bars[S + s]); };
  auto BREADY = [&](int s) { return smem_u32(&bars[2 * S + s]); };
  const uint32_t DONE = smem_u32(&bars[3 * S]);
  auto xst = [&](int s) { return sbase + s * LY::STAGE; };
  auto wst = [&](int s) { return sbase + s * LY::STAGE + kXBytes; };
  auto rawst = [&](int s, int which) { return wst(s) + which * (kChunk * R * 2); };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
      mbar_init(BREADY(s), 4);
    }
    mbar_init(DONE, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), 128);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int n_chunks = d_model / kChunk;
  constexpr uint32_t raw_bytes = (uint32_t)(kChunk * r * 2);

  if (warp == 0) {
    // ------------------------------------------------------------ loads --
    if (lane == 0) {
      int last[S];
      for (int s = 0; s < S; ++s) last[s] = -1;
      // CTAs start at different chunks, so that at any moment they read
      // different rows of A from L2 instead of all the same few lines
      const int rot = (int)(blockIdx.x % (unsigned)n_chunks);
      for (int c = 0; c < n_chunks; ++c) {
        const int s = c % S;
        const int cc = c + rot < n_chunks ? c + rot : c + rot - n_chunks;
        if (c >= S) {
          uint32_t par = (uint32_t)((c / S - 1) & 1);
          if (!mbar_wait(EMPTY(s), par, &abort_flag, errw)) break;
        }
        if (abort_flag) break;
        mbar_expect_tx(FULL(s), kXBytes + 2 * raw_bytes);
        tma_load_2d(xst(s), &xmap, cc * kChunk, t0, FULL(s));
        tma_load_2d(xst(s) + kTile * kBox * 2, &xmap, cc * kChunk + kBox, t0, FULL(s));
        bulk_g2s(rawst(s, 0), Ak + (int64_t)cc * kChunk * r, raw_bytes, FULL(s));
        bulk_g2s(rawst(s, 1), Av + (int64_t)cc * kChunk * r, raw_bytes, FULL(s));
        last[s] = c;
      }
      // copies still in flight land before the CTA may exit
      for (int s = 0; s < S; ++s)
        if (last[s] >= 0 && !mbar_wait_drain(FULL(s), (uint32_t)((last[s] / S) & 1))) abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs --
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, NB, 1);
      for (int c = 0; c < n_chunks; ++c) {
        const int s = c % S;
        uint32_t p1 = (uint32_t)((c / S) & 1), p2 = p1;
        if (!mbar_wait(FULL(s), p1, &abort_flag, errw)) break;
        if (!mbar_wait(BREADY(s), p2, &abort_flag, errw)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) {
          const int b = kk / 4, ks = kk % 4;
          const uint64_t dA = sdesc_sw128(xst(s) + b * (kTile * kBox * 2) + ks * 32);
          const uint64_t dB = sdesc(wst(s) + kk * 2 * NB * 16, NB * 16, 128);
          mma_ss(tmem, dA, dB, idesc, (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(EMPTY(s));
      }
      // tracks every MMA issued above, also after an abort
      mma_commit(DONE);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- transpose B, epilogue --
    const int tw = warp - 2;
    constexpr int gper = r / 8;       // 8-column groups of one of A_k, A_v
    constexpr int kQ = r / 4;         // ldmatrix.x4 per warp and chunk
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % S;
      uint32_t par = (uint32_t)((c / S) & 1);
      const bool ok = mbar_wait(FULL(s), par, &abort_flag, errw);
      // the four warps leave together or not at all (they meet at a named
      // barrier below)
      if (bar_any(!ok || abort_flag)) break;
      // 8x8 blocks (which, kb, gq): rows kb*8.. of the stored chunk, columns
      // gq*8..; instruction q takes blocks 4q .. 4q+3, lane group j = lane/8
      // addresses row lane%8 of block 4q + j.  Every block is read before
      // any is written back (the transpose is in place).
      uint32_t v[kQ][4];
#pragma unroll
      for (int i = 0; i < kQ; ++i) {
        const int q = tw + 4 * i;
        const int bl = q * 4 + (lane >> 3);
        const int which = bl / (16 * gper), rem = bl % (16 * gper);
        const int kb = rem / gper, gq = rem % gper;
        ldsm_x4_t(rawst(s, which) + (uint32_t)((kb * 8 + (lane & 7)) * r * 2 + gq * 16), v[i]);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
      for (int i = 0; i < kQ; ++i) {
        const int q = tw + 4 * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int bj = q * 4 + j;
          const int wj = bj / (16 * gper), rj = bj % (16 * gper);
          const int kbj = rj / gper, gqj = rj % gper;
          // lane holds column nn = gq*8 + lane/4, rows k = kb*8 + 2*(lane%4) + {0, 1}
          const uint32_t off = (uint32_t)(kbj * NB * 16 + (wj * RP + gqj * 8 + (lane >> 2)) * 16 +
                                          (lane & 3) * 4);
          *(uint32_t*)(smem + (wst(s) - sbase) + off) = v[i][j];
        }
      }
      if constexpr (r < RP) {
        // rank-padding columns r .. RP-1 of both halves: 16 x 2 x 8 rows of 16 bytes
        for (int i = tid - 64; i < 16 * 2 * 8; i += 128) {
          const int kb = i / 16, wh = (i / 8) % 2, e = i % 8;
          *(uint4*)(smem + (wst(s) - sbase) + kb * NB * 16 + (wh * RP + r + e) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(BREADY(s));
    }
    uint32_t pd = 0;
    const bool ok = mbar_wait(DONE, pd, &abort_flag, errw) && !abort_flag;
    tc_fence_after();
    if (ok) {
      const int quarter = warp & 3;                    // TMEM lanes this warp may read
      const int row = quarter * 32 + lane, t = pos + t0 + row;
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const bool live = t0 + row < n;
      const int RC = RP / 8;
#pragma unroll
      for (int c0 = 0; c0 < NB; c0 += 32) {
        uint32_t v[32];
        tmem_ld32_wait(tmem + c0 + lane_off, v);
        if (live) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const int nn = c0 + e;                       // 8 columns nn .. nn + 7
            const bool is_v = nn >= RP;
            const int k0 = is_v ? nn - RP : nn;
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
              for (int h = 0; h < 8; ++h)
                vp[h * 8] = (uint16_t)((h & 1) ? (w[h / 2] >> 16) : (w[h / 2] & 0xFFFFu));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // every MMA has completed before TMEM is released (the epilogue's wait
    // may have ended early on an abort)
    if (lane == 0 && !mbar_wait_drain(DONE, 0)) abort_flag = 1;
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <int R>
static int launch_prefill_t(const CUtensorMap& xmap, const PoolGeom& g, uint8_t* lk, uint8_t* lv,
                            int pos, int n, int d_model, const uint16_t* Ak, const uint16_t* Av,
                            cudaStream_t st) {
  using LY = pre::Layout<R>;
  static PerDeviceOnce once;
  const int se = once.run([] {
    return (int)cudaFuncSetAttribute(lr_prefill_kernel<R>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, LY::BYTES);
  });
  if (se != 0) return se;
  const int grid = (n + pre::kTile - 1) / pre::kTile;
  lr_prefill_kernel<R><<<grid, pre::kThreads, LY::BYTES, st>>>(xmap, g, lk, lv, pos, n, d_model,
                                                                Ak, Av);
  return (int)cudaGetLastError();
}

int launch_residual_prefill(const PoolGeom& g, int layer, const AgentDev& ag, int r, int pos, int n,
                            int d_model, const void* x_map, const uint16_t* Ak,
                            const uint16_t* Av, void* stream) {
  uint8_t* lk = g.base + ag.rc_off + (int64_t)layer * rc_layer_bytes(g, ag.rp);
  uint8_t* lv = lk + (int64_t)g.tcap * ag.rp * 2;
  cudaStream_t st = (cudaStream_t)stream;
  CUtensorMap xm;
  std::memcpy(&xm, x_map, sizeof(xm));
  if (ag.rp != (r + 15) / 16 * 16) return (int)cudaErrorInvalidValue;
  switch (r) {
    case 8: return launch_prefill_t<8>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 16: return launch_prefill_t<16>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 24: return launch_prefill_t<24>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 32: return launch_prefill_t<32>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 40: return launch_prefill_t<40>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 48: return launch_prefill_t<48>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 56: return launch_prefill_t<56>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    case 64: return launch_prefill_t<64>(xm, g, lk, lv, pos, n, d_model, Ak, Av, st);
    default: return (int)cudaErrorInvalidValue;
  }
}

}  // namespace fk
