// Skiparse attention backward: the main kernels (the preprocess and post row
// kernels are in skiparse_bwd_rows.cu).
//
// The pages print no backward; it is implied by the method's purpose (it
// accelerates training, "Open-Sora Plan" docs, "Skiparse Attention"). The
// gradient is that of softmax attention inside every scope, followed by the
// transpose of the RoPE rotation for q and k (RoPE came first in the forward).
//
//  preprocess  per token row: delta = rowsum(dO * O) and lse * log2(e) in
//              scope order, rotated bf16 copies of q and k (so the main loop
//              reloads no RoPE), dQ accumulator zeroed, cos/sin table written.
//  main        one work unit = (b, head, scope, 128-row K/V tile); loops over
//              the scope's Q tiles with five tcgen05 MMAs per tile pair:
//                S^T  = K~ Q~^T          dP^T = V dO^T
//                dV  += P^T dO           dK~ += dS^T Q~          dQ~_part = dS K~
//              P^T = exp(S^T * scale - lse), dS^T = P^T * (dP^T - delta).
//              dQ~_part is added into the fp32 accumulator (scope order) by
//              bulk reduce-adds.
//              Epilogue: dv, and dk = scale * R^T dK~, stored at original rows.
//  post        dq = R^T (scale * dQ~_acc) -> bf16.
// One main kernel for D = 128 and D = 64 (18 warps):
//   warps 0-7   P^T / dS^T in four 32-query chunks (one key row, 16 queries of
//               a chunk per thread);
//   warps 8-15  dQ~^T out of TMEM (one channel, 64 queries per thread), staged
//               in the tile's dead Q~ / dO slots and bulk-added to the accumulator;
//               after a unit's last tile, its dK / dV epilogue (one key row,
//               half of the channels per thread), while warps 0-7 start the
//               next unit;
//   warp 16     TMA producer (K~, V per unit; Q~, dO, lse, delta per Q tile);
//   warp 17     MMA issuer; every MMA has M = 128 and N = 128 or D.
// TMEM columns: S^T (P^T as bf16) 0..127, dP^T / dQ~ partial 128..255,
// dV from 256, dK~ from 384 (D columns each).
#include <type_traits>

#include "skiparse_internal.h"

namespace skp {

template <int D>
struct BwdLayout {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int DS_BYTES = 128 * 128 * 2;
  static constexpr int STATS_OFF = 1024;                 // [2 stages][lse2 | delta][128] fp32
  static constexpr int K_OFF = 3072;
  static constexpr int V_OFF = K_OFF + TILE;
  static constexpr int Q_OFF = V_OFF + TILE;            // 2 stages
  static constexpr int DO_OFF = Q_OFF + 2 * TILE;       // 2 stages
  static constexpr int DS_OFF = DO_OFF + 2 * TILE;
  static constexpr int BYTES = DS_OFF + DS_BYTES;
};

__device__ __forceinline__ void decode_unit_bwd(const Geom& g, int u, int& b, int& head, int& s, int& tile) {
  tile = u % g.n_tiles;
  int r = u / g.n_tiles;
  s = g.s0 + (r % g.ks) * g.sstep;               // the ks scopes of this call
  r /= g.ks;
  head = r % g.heads;
  b = r / g.heads;
}

// ===========================================================================
// main kernel (D = 128 and 64): full 128-query tiles, dQ drained by its own warps
// ===========================================================================
//
// Every MMA has M = 128 and N = 128 (N = D for dV and dK~): 40 tcgen05.mma per
// key-tile x query-tile pair at D = 128, 32 at D = 64.
// Per query tile i:
//   MMA1:  S^T = K~ Q~_i^T -> TMEM 0..127, dP^T = V dO_i^T -> TMEM 128..255
//   warps 0-7 form P^T / dS^T in four chunks of 32 queries. P^T of chunks
//          0 and 1 is published as soon as S^T lands (while dP^T is still on
//          the tensor core), so dV += P^T_{0,1} dO_i[0:64] runs while the warps
//          form dS^T_0; after each dS^T_c the tensor core runs dK~ += dS^T_c
//          Q~_i[c] (and dV for chunks 2, 3) while the warps form chunk c+1;
//   MMA3:  dQ~^T = K~^T dS^T -> TMEM 128..255 (M = 128 channels, N = 128 queries)
// Warps 8-15 copy dQ~^T out of TMEM (one channel, 64 queries per thread),
// release it, stage it in the tile's own Q~ / dO slots (dead by then until the
// refill two tiles later) and add it into the scope-order fp32 accumulator with
// two bulk reduce-adds, which the TMA engine streams to L2 while the next tile
// runs. (Reduction stores issued from registers would instead share the
// load/store pipe with the softmax warps' shared-memory traffic and slow it.)
// P^T for queries 16m .. 16m+15 is packed into S^T columns 16m .. 16m+7, which
// the writing thread has itself read; warps w and w+4 share TMEM lanes (key
// rows) and split each chunk's 32 queries 16 / 16.
enum BwdTileBar {
  T_KVFULL, T_KVEMPTY,
  T_QFULL0, T_QFULL1,       // Q~ tile + lse / delta of stage 0 / 1 landed
  T_OFULL0, T_OFULL1,       // dO tile of stage 0 / 1 landed
  T_QFREE0, T_QFREE1,       // Q~ slot of stage 0 / 1 free again (its dQ~ staging has been read)
  T_OFREE0, T_OFREE1,       // dO slot likewise
  T_SRDY, T_DPRDY, T_PRDY, T_DSC0, T_DSC1, T_DSC2, T_DSC3, T_DQFULL, T_DQFREE, T_DKVDONE, T_DVFREE, T_DKFREE, T_FINAL,
  T_NBARS
};

constexpr int kTileThreads = 576;   // 8 softmax warps, 8 dQ warps, TMA warp, MMA warp
constexpr int kTileTmaWarp = 16, kTileMmaWarp = 17;

// Query tile visited at step i by the unit of key tile kt. The CTAs of one
// scope start together; rotating the order by kt spreads their dQ~ adds over
// different accumulator rows.
__device__ __forceinline__ int stagger(int i, int kt, int n) {
  const int r = i + kt;
  return r >= n ? r - n : r;
}

template <int D>
__global__ void __launch_bounds__(kTileThreads, 1) skiparse_bwd_main_tile_kernel(const __grid_constant__ BwdParams p) {
  using Ly = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) atomicCAS(p.err, 0, ERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  int* abort_flag = reinterpret_cast<int*>(smem + 520);
  float* stats = reinterpret_cast<float*>(smem + Ly::STATS_OFF);
  const uint32_t sK = smem_u32(smem + Ly::K_OFF);
  const uint32_t sV = smem_u32(smem + Ly::V_OFF);
  const uint32_t sQ = smem_u32(smem + Ly::Q_OFF);
  const uint32_t sDO = smem_u32(smem + Ly::DO_OFF);
  const uint32_t sDS = smem_u32(smem + Ly::DS_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const Ctl ctl{abort_flag, p.err};
  const Geom& g = p.g;
  constexpr int E = ERR_KERNEL_BWD + 0x80;

  if (tid == 0) {
    *abort_flag = 0;
    const uint32_t counts[T_NBARS] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 8, 8, 8, 8, 8, 1, 8, 1, 8, 8, 1};
    for (int i = 0; i < T_NBARS; ++i) mbar_init(bar(i), counts[i]);
    mbar_fence_init();
  }
  if (warp == kTileMmaWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The TMA and MMA warps run their loops with all 32 lanes (waits are voted
  // across the warp so every lane takes the same branch); lane 0 issues.
  auto warp_wait = [&](int i, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ctl, E + i)) != 0;
  };
  const bool leader = lane == 0;
  if (warp == kTileTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (leader) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      tma_prefetch_map(&p.tm_do);
    }
    uint32_t kv_issued = 0, q_issued[2] = {0, 0};
    uint32_t g0 = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int b, head, s, kt;
      decode_unit_bwd(g, u, b, head, s, kt);
      const int nt = scope_tiles(g, s);
      if (kt >= nt) continue;                         // a shorter scope has fewer key tiles
      if (it > 0 && !warp_wait(T_KVEMPTY, (it - 1) & 1)) break;
      if (leader) {
        mbar_expect_tx(bar(T_KVFULL), 2 * Ly::TILE);
        const TileCoord tck = scope_tile(g, s, b, kt * kTile);
#pragma unroll
        for (int h = 0; h < Ly::HALVES; ++h) {
          load_tile(sK + h * kHalfBytes, &p.tm_k, bar(T_KVFULL), tck, h * 64, head);
          load_tile(sV + h * kHalfBytes, &p.tm_v, bar(T_KVFULL), tck, h * 64, head);
        }
      }
      __syncwarp();
      ++kv_issued;
      const size_t srow = (((size_t)b * g.heads + head) * g.k + s) * p.Lp;
      for (int i = 0; i < nt; ++i) {
        const uint32_t gg = g0 + i;
        const int st = gg & 1;
        const uint32_t n = gg >> 1;
        const int qi = stagger(i, kt, nt);
        const TileCoord tcq = scope_tile(g, s, b, qi * kTile);   // before the slot waits
        // a slot is refilled once the dQ~ staging of tile gg-2 placed in it has been read out
        if (n > 0 && !warp_wait(T_QFREE0 + st, (n - 1) & 1)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(bar(T_QFULL0 + st), Ly::TILE + 1024);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            load_tile(sQ + st * Ly::TILE + h * kHalfBytes, &p.tm_q, bar(T_QFULL0 + st), tcq, h * 64, head);
          const uint32_t dst = smem_u32(stats + st * 256);
          bulk_load(dst, p.lse2s + srow + qi * kTile, 512, bar(T_QFULL0 + st));
          bulk_load(dst + 512, p.delta_s + srow + qi * kTile, 512, bar(T_QFULL0 + st));
        }
        __syncwarp();
        if (n > 0 && !warp_wait(T_OFREE0 + st, (n - 1) & 1)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_expect_tx(bar(T_OFULL0 + st), Ly::TILE);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            load_tile(sDO + st * Ly::TILE + h * kHalfBytes, &p.tm_do, bar(T_OFULL0 + st), tcq, h * 64, head);
        }
        __syncwarp();
        ++q_issued[st];
      }
      g0 += nt;
      ++it;
    }
    if (leader) {
      if (kv_issued) mbar_drain(bar(T_KVFULL), (kv_issued - 1) & 1);
      for (int st = 0; st < 2; ++st)
        if (q_issued[st]) {
          mbar_drain(bar(T_QFULL0 + st), (q_issued[st] - 1) & 1);
          mbar_drain(bar(T_OFULL0 + st), (q_issued[st] - 1) & 1);
        }
    }
    __syncwarp();
  } else if (warp == kTileMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);   // S^T, dP^T
    constexpr uint32_t kIdDV = idesc_bf16(128, D, false, true);     // P^T (TMEM) x dO (MN-major)
    constexpr uint32_t kIdDK = idesc_bf16(128, D, false, true);     // dS^T (K-major) x Q~ (MN-major)
    // dQ~^T = K~^T dS^T: M = 128 channel rows, N = 128 queries. With D = 64 the
    // A operand's second 64-row block is the V tile (the next 16 KB): rows 64-127
    // of the product are not used (an M = 64 product would take as many MMAs)
    constexpr uint32_t kIdDQ = idesc_bf16(128, 128, true, true);      // K~^T (MN-major) x dS^T (MN-major)
    // k-step-0 descriptors of every operand tile; k-steps add a constant
    const uint64_t dKk = desc_kmajor(sK, 0), dKmn = desc_mnmajor(sK, 0), dVk = desc_kmajor(sV, 0);
    const uint64_t dDSk = desc_kmajor(sDS, 0), dDSmn = desc_mnmajor(sDS, 0);
    uint32_t g0 = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int b, head, s, kt;
      decode_unit_bwd(g, u, b, head, s, kt);
      const int nt = scope_tiles(g, s);
      if (kt >= nt) continue;
      if (!warp_wait(T_KVFULL, it & 1)) break;
      tc_fence_after();
      for (int i = 0; ok && i < nt; ++i) {
        const uint32_t gg = g0 + i;
        const int st = gg & 1;
        if (!warp_wait(T_QFULL0 + st, (gg >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qt = sQ + st * Ly::TILE;
        const uint32_t dot = sDO + st * Ly::TILE;
        const uint64_t dQk = desc_kmajor(qt, 0), dQmn = desc_mnmajor(qt, 0);
        const uint64_t dOk = desc_kmajor(dot, 0), dOmn = desc_mnmajor(dot, 0);
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss(tmem, kmajor_step(dKk, ks), kmajor_step(dQk, ks), kIdS, ks > 0 ? 1u : 0u);
          tc_commit(bar(T_SRDY));
        }
        __syncwarp();
        // dP^T overwrites the previous tile's dQ~^T: wait until the dQ warps hold it
        if (gg > 0 && !warp_wait(T_DQFREE, (gg - 1) & 1)) { ok = false; break; }
        if (!warp_wait(T_OFULL0 + st, (gg >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_ss(tmem + 128, kmajor_step(dVk, ks), kmajor_step(dOk, ks), kIdS, ks > 0 ? 1u : 0u);
          tc_commit(bar(T_DPRDY));
        }
        __syncwarp();
        // P^T of queries 0..63 is published while dP^T is still being computed
        if (!warp_wait(T_PRDY, gg & 1)) { ok = false; break; }
        // the previous unit's dV must have been read out of TMEM before the first accumulate
        if (i == 0 && it > 0 && !warp_wait(T_DVFREE, (it - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ts(tmem + 256, tmem + 16 * ks, mnmajor_step(dOmn, ks), kIdDV, (i > 0 || ks > 0) ? 1u : 0u);
        }
        __syncwarp();
        for (int c = 0; c < 4; ++c) {
          if (!warp_wait(T_DSC0 + c, gg & 1)) { ok = false; break; }
          // likewise the previous unit's dK~ before the first dK~ accumulate
          if (c == 0 && i == 0 && it > 0 && !warp_wait(T_DKFREE, (it - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          if (leader) {
            if (c >= 2) {
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int ks = 2 * c + e;
                mma_ts(tmem + 256, tmem + 16 * ks, mnmajor_step(dOmn, ks), kIdDV, 1u);
              }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int ks = 2 * c + e;
              mma_ss(tmem + 384, kmajor_step(dDSk, ks), mnmajor_step(dQmn, ks), kIdDK, (i > 0 || ks > 0) ? 1u : 0u);
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(tmem + 128, mnmajor_step(dKmn, ks), mnmajor_step(dDSmn, ks), kIdDQ, ks > 0 ? 1u : 0u);
          tc_commit(bar(T_DQFULL));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) {
        tc_commit(bar(T_DKVDONE));
        tc_commit(bar(T_KVEMPTY));
      }
      __syncwarp();
      g0 += nt;
      ++it;
    }
    if (leader) {
      tc_commit(bar(T_FINAL));
      mbar_drain(bar(T_FINAL), 0);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ warps (8-15)
    // Tile gg's Q~ and dO slots are dead once DQFULL(gg) fired (it follows the
    // last MMA reading them) and stay so until the tile gg+2 refill: the two
    // query halves of dQ~ are staged there as 64 x 128 fp32 row blocks and
    // bulk-added into the accumulator; the slot is released when read out.
    const int j = (warp & 3) * 32 + lane;                    // channel d = TMEM lane of dQ~^T
    const int qh = (warp - 8) >> 2;                          // query half: 0 -> Q~ slot, 1 -> dO slot
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool leader = tid == 256;
    uint32_t g0 = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int b, head, s, kt;
      decode_unit_bwd(g, u, b, head, s, kt);
      const int nt = scope_tiles(g, s);
      if (kt >= nt) continue;
      float* acc = p.dq_acc + (((size_t)b * g.heads + head) * g.k + s) * (size_t)p.Lp * D;
      for (int i = 0; i < nt; ++i) {
        const uint32_t gg = g0 + i;
        const int st = gg & 1;
        if (!bar_and<3, 256>(mbar_wait(bar(T_DQFULL), gg & 1, ctl, E + T_DQFULL))) { ok = false; break; }
        tc_fence_after();
        float x[64];
        tmem_ld32(tmem + lane_base + 128 + qh * 64, *reinterpret_cast<float(*)[32]>(&x[0]));
        tmem_ld32(tmem + lane_base + 128 + qh * 64 + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(T_DQFREE));
        float* slot = reinterpret_cast<float*>(smem + (qh ? Ly::DO_OFF : Ly::Q_OFF) + st * Ly::TILE);
        if (D == 128 || j < D) {                       // D = 64: TMEM lanes 64-127 hold unused rows
#pragma unroll
          for (int q = 0; q < 64; ++q) slot[q * D + j] = x[q];
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 4, 256;" ::: "memory");
        if (leader) {
          // the Q~ slot's half first: Q~ of tile gg+2 is needed before its dO
          const int q0 = stagger(i, kt, nt) * kTile;   // rows < Lp: padded rows get zeros
          bulk_reduce_add_f32(acc + (size_t)q0 * D, smem_u32(smem + Ly::Q_OFF + st * Ly::TILE), 64 * D * 4);
          bulk_commit_group();
          bulk_reduce_add_f32(acc + (size_t)(q0 + 64) * D, smem_u32(smem + Ly::DO_OFF + st * Ly::TILE), 64 * D * 4);
          bulk_commit_group();
          bulk_wait_read<1>();
          mbar_arrive(bar(T_QFREE0 + st));
          bulk_wait_read<0>();
          mbar_arrive(bar(T_OFREE0 + st));
        }
        __syncwarp();
      }
      if (!ok) break;
      const int jr = (warp & 3) * 32 + lane;             // key row (TMEM lane)
      const bool key_ok = kt * kTile + jr < scope_len(g, s);
      // ---- epilogue of the unit (these warps wait for the next unit's first dQ~
      // anyway; the softmax warps go straight on): dv, and dk = scale * R^T dK~
      // (key row jr; the two warps on a row share the chunks out)
      if (!bar_and<3, 256>(mbar_wait(bar(T_DKVDONE), it & 1, ctl, E + T_DKVDONE))) break;
      tc_fence_after();
      const int prow = kt * kTile + jr;
      const int tok = key_ok ? token_of(g, s, prow) : 0;
      int t = 0, hh = 0, w = 0;
      if (key_ok) token_coords(p.rope, tok, t, hh, w);
      const size_t rbase = (((size_t)b * g.N + tok) * g.heads + head) * D;
      // Each of the two warps on a key row writes half of dv and half of dk: the
      // dk chunks' cos / sin reads (scattered over the tokens of the warp's 32
      // key rows, the w axis worst) are shared out, chunks 0 + 3 and 1 + 2.
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = qh * (D / 64) + cc;              // dv chunks 0, 1 / 2, 3 (D = 64: 0 / 1)
        float y[32];
        tmem_ld32(tmem + lane_base + 256 + c * 32, y);
        if (key_ok) {
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = pack_bf16(y[2 * e], y[2 * e + 1]);
          // rows are D * 2 bytes apart: 32-byte stores whenever the base allows
          st_global_64b(p.dv + rbase + c * 32, o, (reinterpret_cast<uintptr_t>(p.dv) & 31u) == 0);
        }
      }
      // dV is out of TMEM: the next unit's first P^T dO may start while dk is formed
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(T_DVFREE));
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = D == 128 ? (qh == 0 ? 3 * cc : 1 + cc) : qh + 2 * cc;   // dk chunks 0, 3 / 1, 2
        if (c >= D / 32) break;
        float y[32];
        tmem_ld32(tmem + lane_base + 384 + c * 32, y);
        if (key_ok) {
          // pairs 16c .. 16c + 15, two per 16-byte table read (an axis never
          // splits a pair of pairs: its bounds D/8 and 5D/16 are even)
          float4 cs[8];
#pragma unroll
          for (int e2 = 0; e2 < 8; ++e2) {
            const PairSel sel = pair_select(p.rope, c * 16 + 2 * e2);
            cs[e2] = __ldg(reinterpret_cast<const float4*>(&p.rope_tab[pair_index(sel, t, hh, w)]));
          }
          uint32_t o[16];
#pragma unroll
          for (int e2 = 0; e2 < 8; ++e2) {
            const float2 r0 = rope_rotate_t(y[4 * e2] * p.scale, y[4 * e2 + 1] * p.scale,
                                            make_float2(cs[e2].x, cs[e2].y));
            const float2 r1 = rope_rotate_t(y[4 * e2 + 2] * p.scale, y[4 * e2 + 3] * p.scale,
                                            make_float2(cs[e2].z, cs[e2].w));
            o[2 * e2] = pack_bf16(r0.x, r0.y);
            o[2 * e2 + 1] = pack_bf16(r1.x, r1.y);
          }
          st_global_64b(p.dk + rbase + c * 32, o, (reinterpret_cast<uintptr_t>(p.dk) & 31u) == 0);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(T_DKFREE));
      g0 += nt;
      ++it;
    }
    if (leader) bulk_wait_all();
  } else {
    // ------------------------------------------------------------ P^T / dS^T warps (0-7)
    const int ch = warp >> 2;                                // which 16 queries of each 32-query chunk
    const int j = (warp & 3) * 32 + lane;                    // key row (TMEM lane)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* ds_row = smem + Ly::DS_OFF + j * 128;
    uint32_t g0 = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int b, head, s, kt;
      decode_unit_bwd(g, u, b, head, s, kt);
      const int nt = scope_tiles(g, s);
      if (kt >= nt) continue;
      const int Ls = scope_len(g, s);
      const bool key_ok = kt * kTile + j < Ls;
      for (int i = 0; i < nt; ++i) {
        const uint32_t gg = g0 + i;
        const int st = gg & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(T_SRDY), gg & 1, ctl, E + T_SRDY))) { ok = false; break; }
        tc_fence_after();
        const float4* lse4 = reinterpret_cast<const float4*>(stats + st * 256);
        const float4* del4 = lse4 + 32;
        const int qvalid = key_ok ? min(kTile, Ls - stagger(i, kt, nt) * kTile) : 0;
        // Full tiles (every key row of the warp and every query of the tile inside
        // the scope: all but the last query or key tile) take a select-free path;
        // rows and columns past the scope are zeroed otherwise. Warp-uniform, so
        // both paths keep their warp-level synchronisation.
        const bool full = __all_sync(0xffffffffu, qvalid == kTile) != 0;
        const unsigned long long sl2x2 = f2_pack(sl2, sl2);
        // P = exp2(S * scale * log2(e) - lse * log2(e)) for this thread's 16 queries at qb
        auto exp_p = [&](auto F, const float (&sv)[16], int qb, float (&pv)[16]) {
          constexpr bool FULL = decltype(F)::value;
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 l4 = lse4[(qb >> 2) + e4];
            float a[4];
            f2_unpack(ffma2(f2_pack(sv[e4 * 4], sv[e4 * 4 + 1]), sl2x2, f2_pack(-l4.x, -l4.y)), a[0], a[1]);
            f2_unpack(ffma2(f2_pack(sv[e4 * 4 + 2], sv[e4 * 4 + 3]), sl2x2, f2_pack(-l4.z, -l4.w)), a[2], a[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float pe = ex2(a[e]);
              pv[e4 * 4 + e] = (FULL || qb + e4 * 4 + e < qvalid) ? pe : 0.f;
            }
          }
        };
        auto store_pt = [&](const float (&pv)[16], int qb) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_bf16(pv[2 * e], pv[2 * e + 1]);
          // P^T over this thread's own S^T columns qb .. qb+7 (already read by this thread)
          tmem_st8(tmem + lane_base + qb, pk);
        };
        // dS^T = P^T * (dP^T - delta) -> row j of the dS^T buffer, queries qb .. qb+15
        // (explicit zero past the scope: the padded delta entries are never written)
        auto store_ds = [&](auto F, const float (&pv)[16], const float (&dp)[16], int c, int qb) {
          constexpr bool FULL = decltype(F)::value;
          uint32_t dk[8];
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 d4 = del4[(qb >> 2) + e4];
            float dsv[4];
            f2_unpack(fmul2(f2_pack(pv[e4 * 4], pv[e4 * 4 + 1]),
                            fsub2(f2_pack(dp[e4 * 4], dp[e4 * 4 + 1]), f2_pack(d4.x, d4.y))), dsv[0], dsv[1]);
            f2_unpack(fmul2(f2_pack(pv[e4 * 4 + 2], pv[e4 * 4 + 3]),
                            fsub2(f2_pack(dp[e4 * 4 + 2], dp[e4 * 4 + 3]), f2_pack(d4.z, d4.w))), dsv[2], dsv[3]);
            if (!FULL) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (qb + e4 * 4 + e >= qvalid) dsv[e] = 0.f;
            }
            dk[e4 * 2] = pack_bf16(dsv[0], dsv[1]);
            dk[e4 * 2 + 1] = pack_bf16(dsv[2], dsv[3]);
          }
          // box c/2, 16-byte chunks (c%2)*4 + ch*2 + {0,1}
          uint8_t* rowp = ds_row + (c >> 1) * kHalfBytes;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int chunk = ((c & 1) * 4 + ch * 2 + q2) ^ (j & 7);
            *reinterpret_cast<uint4*>(rowp + chunk * 16) = make_uint4(dk[4 * q2], dk[4 * q2 + 1], dk[4 * q2 + 2], dk[4 * q2 + 3]);
          }
        };
        // chunks 0 and 1: P^T first (the tensor core computes dP^T meanwhile), P kept in fp32
        float p01[2][16];
        auto p_phase = [&](auto F) {
          float s0[16], s1[16];
          tmem_ld16x2(tmem + lane_base + ch * 16, tmem + lane_base + 32 + ch * 16, s0, s1);
          exp_p(F, s0, ch * 16, p01[0]);
          exp_p(F, s1, 32 + ch * 16, p01[1]);
          store_pt(p01[0], ch * 16);
          store_pt(p01[1], 32 + ch * 16);
        };
        if (full) p_phase(std::true_type{});
        else p_phase(std::false_type{});
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(T_PRDY));
        // DPRDY also says the previous tile's MMAs (readers of the dS^T buffer) are done
        if (!__all_sync(0xffffffffu, mbar_wait(bar(T_DPRDY), gg & 1, ctl, E + T_DPRDY))) { ok = false; break; }
        tc_fence_after();
        auto ds_phase = [&](auto F) {
          // dP^T of chunks 0 and 1 in one TMEM round trip
          float dp01[2][16];
          tmem_ld16x2(tmem + lane_base + 128 + ch * 16, tmem + lane_base + 128 + 32 + ch * 16, dp01[0], dp01[1]);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            store_ds(F, p01[c], dp01[c], c, c * 32 + ch * 16);
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T_DSC0 + c));
          }
#pragma unroll
          for (int c = 2; c < 4; ++c) {
            const int qb = c * 32 + ch * 16;
            float sv[16], dp[16], pv[16];
            tmem_ld16x2(tmem + lane_base + qb, tmem + lane_base + 128 + qb, sv, dp);
            exp_p(F, sv, qb, pv);
            store_pt(pv, qb);
            store_ds(F, pv, dp, c, qb);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T_DSC0 + c));
          }
        };
        if (full) ds_phase(std::true_type{});
        else ds_phase(std::false_type{});
      }
      if (!ok) break;
      g0 += nt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTileMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t bwd_main_smem_bytes(int D) {
  return D == 128 ? (size_t)BwdLayout<128>::BYTES : (size_t)BwdLayout<64>::BYTES;
}

template <int D>
static cudaError_t launch_tile(const BwdParams& p, int grid, cudaStream_t stream) {
  const cudaError_t e = cudaFuncSetAttribute(skiparse_bwd_main_tile_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bwd_main_smem_bytes(D));
  if (e != cudaSuccess) return e;
  skiparse_bwd_main_tile_kernel<D><<<grid, kTileThreads, bwd_main_smem_bytes(D), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, int grid, cudaStream_t stream) {
  return p.g.D == 128 ? launch_tile<128>(p, grid, stream) : launch_tile<64>(p, grid, stream);
}

}  // namespace skp
