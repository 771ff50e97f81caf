// Skiparse attention forward: one persistent kernel per call.
//
// What it computes ("Open-Sora Plan" docs, "Skiparse Attention", single and
// group skip listings): for every (batch b, head, scope s) the softmax
// attention of the scope's L = N/k tokens among themselves, with q and k
// rotated by 3D RoPE at their original positions, written back to the tokens'
// original rows. The rearrange never happens in memory: the TMA tensor maps
// address the scope's rows directly (see skiparse_host.cu), and the epilogue
// stores each output row at its original token index.
//
// One work unit = (b, head, s, a pair of 128-row Q tiles A and B), so every
// K / V tile is loaded and rotated once for 256 query rows. Warp roles:
//   warps 0-3   softmax for Q tile A, one query row per thread (TMEM lane);
//   warps 4-7   softmax for Q tile B;
//   warps 8-11  RoPE: rotate the Q tiles and each K tile in shared memory
//               (16-byte chunks, per-row table offsets staged in shared memory);
//   warp  12    TMA producer: Q pair, then a 2-stage K / V ring;
//   warp  13    MMA issuer (tcgen05.mma kind::f16, fp32 accumulators in TMEM).
// TMEM columns: S_A / P_A 0..127, S_B / P_B 128..255, O_A 256.., O_B 384...
// MMA issue order: S_A(g), S_B(g), PV_A(g), S_A(g+1), PV_B(g), S_B(g+1), ...
// so each softmax warpgroup's critical loop is softmax + two MMA groups while
// the tensor core alternates between the two Q tiles. Because S_X(g) is issued
// after PV_X(g-1), the S-full barrier of tile g proves PV_X(g-1) complete, which
// keeps every parity wait on the O-done barriers one phase ahead at most.
// The softmax reads S twice from TMEM (max pass, then exp pass) so that all 14
// warps fit in 128 registers; online softmax with lazy O rescaling (threshold
// 2^8), P written back over S as bf16.
#include "skiparse_internal.h"

namespace skp {

template <int D>
struct FwdLayout {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int HDR = 1024;
  static constexpr int QA_OFF = HDR;
  static constexpr int QB_OFF = QA_OFF + TILE;
  static constexpr int K_OFF = QB_OFF + TILE;
  static constexpr int V_OFF = K_OFF + 2 * TILE;
  static constexpr int ROWOFF_OFF = V_OFF + 2 * TILE;   // [2][128] int4 per-row RoPE table offsets
  static constexpr int ROPE_OFF = ROWOFF_OFF + 2 * 128 * 16;
};

enum FwdBar {
  F_QFULL, F_QROT, F_QEMPTY,
  F_KFULL0, F_KFULL1, F_KROT0, F_KROT1, F_KEMPTY0, F_KEMPTY1,
  F_VFULL0, F_VFULL1, F_VEMPTY0, F_VEMPTY1,
  F_SFULL_A, F_SFULL_B, F_PFULL_A, F_PFULL_B, F_ODONE_A, F_ODONE_B, F_OEMPTY_A, F_OEMPTY_B, F_FINAL, F_NBARS
};

constexpr int kFwdThreads = 448;

__device__ __forceinline__ void decode_unit(const Geom& g, int n_pairs, int u, int& b, int& head, int& s, int& pair) {
  pair = u % n_pairs;
  int r = u / n_pairs;
  s = r % g.k;
  r /= g.k;
  head = r % g.heads;
  b = r / g.heads;
}

// Named barrier over the 4 RoPE warps that also ANDs a predicate across them,
// so that every RoPE warp takes the same branch after a bounded wait.
__device__ __forceinline__ bool rope_bar_and(bool v) {
  uint32_t out;
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(out) : "r"(v ? 1u : 0u) : "memory");
  return out != 0;
}

// Rotate the rows of one 128-row tile in shared memory, in place. The tile
// holds positions p0 .. p0+127 of scope s; rows at or past L are left alone.
// Step 1: RoPE thread r (0..127) stores row r's table offsets in `rowoff`
// (entry of pair 0 of the t, h and w chunks at the row's position, and a
// valid flag). Step 2, after the barrier (which also ANDs `ok`): a lane owns
// one 16-byte chunk (4 channel pairs, always inside one axis chunk) of one of
// 4 rows, so a warp touches 4 whole 128-byte rows per step. Returns false if
// any RoPE thread passed in ok = false (then nothing is rotated).
template <int D>
__device__ __forceinline__ bool rope_tile(uint8_t* tile, int4* rowoff, int p0, int s, const Geom& g,
                                          const RopeParams& rp, const float2* tab, int rtid, int lane, bool ok) {
  constexpr int HALVES = D / 64;
  {
    const int p = p0 + rtid;
    int4 ro = make_int4(0, 0, 0, 0);
    if (ok && p < g.L) {
      int t, hh, w;
      token_coords(rp, token_of(g, s, p), t, hh, w);
      const int bt = rp.T * rp.dt2;
      ro = make_int4(t * rp.dt2, bt + hh * rp.dh2, bt + rp.H * rp.dh2 + w * rp.dh2, 1);
    }
    rowoff[rtid] = ro;
  }
  if (!rope_bar_and(ok)) return false;
  const int wid = rtid >> 5;
  const int rsub = lane >> 3;
  const int c = lane & 7;
  int axis[HALVES], local[HALVES];
#pragma unroll
  for (int hb = 0; hb < HALVES; ++hb) {
    const PairSel sel = pair_select(rp, (hb * 8 + c) * 4);
    axis[hb] = sel.axis;
    local[hb] = sel.local;
  }
#pragma unroll 2
  for (int it = 0; it < 8; ++it) {
    const int r = wid * 32 + it * 4 + rsub;
    const int4 ro = rowoff[r];
    if (!ro.w) continue;
#pragma unroll
    for (int hb = 0; hb < HALVES; ++hb) {
      const int e = (axis[hb] == 0 ? ro.x : (axis[hb] == 1 ? ro.y : ro.z)) + local[hb];
      const float4 cs01 = *reinterpret_cast<const float4*>(tab + e);
      const float4 cs23 = *reinterpret_cast<const float4*>(tab + e + 2);
      uint4* ptr = reinterpret_cast<uint4*>(tile + hb * kHalfBytes + r * 128 + ((c ^ (r & 7)) << 4));
      const uint4 v = *ptr;
      const float2 a0 = rope_rotate(bf16lo(v.x), bf16hi(v.x), make_float2(cs01.x, cs01.y));
      const float2 a1 = rope_rotate(bf16lo(v.y), bf16hi(v.y), make_float2(cs01.z, cs01.w));
      const float2 a2 = rope_rotate(bf16lo(v.z), bf16hi(v.z), make_float2(cs23.x, cs23.y));
      const float2 a3 = rope_rotate(bf16lo(v.w), bf16hi(v.w), make_float2(cs23.z, cs23.w));
      *ptr = make_uint4(pack_bf16(a0.x, a0.y), pack_bf16(a1.x, a1.y), pack_bf16(a2.x, a2.y), pack_bf16(a3.x, a3.y));
    }
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(512, 1) skiparse_fwd_kernel(const __grid_constant__ FwdParams p) {
  using Ly = FwdLayout<D>;
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
  float2* tab = reinterpret_cast<float2*>(smem + Ly::ROPE_OFF);
  int4* rowoff = reinterpret_cast<int4*>(smem + Ly::ROWOFF_OFF);
  const uint32_t sQA = smem_u32(smem + Ly::QA_OFF);
  const uint32_t sQB = smem_u32(smem + Ly::QB_OFF);
  const uint32_t sK = smem_u32(smem + Ly::K_OFF);
  const uint32_t sV = smem_u32(smem + Ly::V_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const Ctl ctl{abort_flag, p.err};
  const Geom& g = p.g;
  const int n_pairs = (g.n_tiles + 1) >> 1;

  if (tid == 0) {
    *abort_flag = 0;
    const uint32_t counts[F_NBARS] = {1, 4, 1, 1, 1, 4, 4, 1, 1, 1, 1, 1, 1, 1, 1, 4, 4, 1, 1, 4, 4, 1};
    for (int i = 0; i < F_NBARS; ++i) mbar_init(bar(i), counts[i]);
    mbar_fence_init();
  }
  if (warp == 13) tmem_alloc(smem_u32(tmem_slot), 512);
  rope_build_table(tab, p.rope, tid, kFwdThreads);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      uint32_t q_issued = 0, k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
      uint32_t gk = 0;
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++it) {
        int b, head, s, pair;
        decode_unit(g, n_pairs, u, b, head, s, pair);
        if (it > 0 && !mbar_wait(bar(F_QEMPTY), (it - 1) & 1, ctl, ERR_KERNEL_FWD + F_QEMPTY)) break;
        mbar_expect_tx(bar(F_QFULL), 2 * Ly::TILE);
        const int qrow = b * g.Nn + (2 * pair * kTile) / g.G;
#pragma unroll
        for (int h = 0; h < Ly::HALVES; ++h) {
          tma_load_5d(sQA + h * kHalfBytes, &p.tm_q, bar(F_QFULL), h * 64, head, 0, s, qrow);
          tma_load_5d(sQB + h * kHalfBytes, &p.tm_q, bar(F_QFULL), h * 64, head, 0, s, qrow + kTile / g.G);
        }
        ++q_issued;
        for (int j = 0; j < g.n_tiles; ++j) {
          const uint32_t gg = gk + j;
          const int st = gg & 1;
          const uint32_t n = gg >> 1;
          const int krow = b * g.Nn + (j * kTile) / g.G;
          if (n > 0 && !mbar_wait(bar(F_KEMPTY0 + st), (n - 1) & 1, ctl, ERR_KERNEL_FWD + F_KEMPTY0 + st)) { ok = false; break; }
          mbar_expect_tx(bar(F_KFULL0 + st), Ly::TILE);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            tma_load_5d(sK + st * Ly::TILE + h * kHalfBytes, &p.tm_k, bar(F_KFULL0 + st), h * 64, head, 0, s, krow);
          ++k_issued[st];
          if (n > 0 && !mbar_wait(bar(F_VEMPTY0 + st), (n - 1) & 1, ctl, ERR_KERNEL_FWD + F_VEMPTY0 + st)) { ok = false; break; }
          mbar_expect_tx(bar(F_VFULL0 + st), Ly::TILE);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            tma_load_5d(sV + st * Ly::TILE + h * kHalfBytes, &p.tm_v, bar(F_VFULL0 + st), h * 64, head, 0, s, krow);
          ++v_issued[st];
        }
        gk += g.n_tiles;
      }
      // Copies still in flight (only after an abort) must land before exit.
      if (q_issued) mbar_drain(bar(F_QFULL), (q_issued - 1) & 1);
      for (int st = 0; st < 2; ++st) {
        if (k_issued[st]) mbar_drain(bar(F_KFULL0 + st), (k_issued[st] - 1) & 1);
        if (v_issued[st]) mbar_drain(bar(F_VFULL0 + st), (v_issued[st] - 1) & 1);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
      uint32_t g0 = 0;
      int it = 0;
      bool ok = true;
      // S_X = Q_X K_g^T into TMEM columns colS (X = A: 0, B: 128)
      auto issue_s = [&](uint32_t qt, uint32_t colS, int st) {
        const uint32_t kt = sK + st * Ly::TILE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + colS, desc_kmajor(qt, ks), desc_kmajor(kt, ks), kIdS, ks > 0 ? 1u : 0u);
      };
      // O_X += P_X V_g, P_X in TMEM over S_X
      auto issue_pv = [&](uint32_t colS, uint32_t colO, int st, bool first) {
        const uint32_t vt = sV + st * Ly::TILE;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tmem + colO, tmem + colS + ks * 8, desc_mnmajor(vt, ks), kIdPV, (!first || ks > 0) ? 1u : 0u);
      };
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++it) {
        const int n = g.n_tiles;
        if (!mbar_wait(bar(F_QROT), it & 1, ctl, ERR_KERNEL_FWD + F_QROT)) break;
        if (!mbar_wait(bar(F_KROT0 + (g0 & 1)), (g0 >> 1) & 1, ctl, ERR_KERNEL_FWD + F_KROT0)) break;
        tc_fence_after();
        issue_s(sQA, 0, g0 & 1);
        tc_commit(bar(F_SFULL_A));
        issue_s(sQB, 128, g0 & 1);
        tc_commit(bar(F_SFULL_B));
        tc_commit(bar(F_KEMPTY0 + (g0 & 1)));
        if (n == 1) tc_commit(bar(F_QEMPTY));
        for (int j = 0; j < n; ++j) {
          const uint32_t gg = g0 + j;
          const int st = gg & 1;
          const uint32_t nn = gg >> 1;
          // PV_A(g)
          if (j == 0 && it > 0 && !mbar_wait(bar(F_OEMPTY_A), (it - 1) & 1, ctl, ERR_KERNEL_FWD + F_OEMPTY_A)) { ok = false; break; }
          if (!mbar_wait(bar(F_PFULL_A), gg & 1, ctl, ERR_KERNEL_FWD + F_PFULL_A)) { ok = false; break; }
          if (!mbar_wait(bar(F_VFULL0 + st), nn & 1, ctl, ERR_KERNEL_FWD + F_VFULL0 + st)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, 256, st, j == 0);
          tc_commit(bar(F_ODONE_A));
          // S_A(g+1)
          const bool more = j + 1 < n;
          if (more) {
            const int st1 = (gg + 1) & 1;
            if (!mbar_wait(bar(F_KROT0 + st1), ((gg + 1) >> 1) & 1, ctl, ERR_KERNEL_FWD + F_KROT0 + st1)) { ok = false; break; }
            tc_fence_after();
            issue_s(sQA, 0, st1);
            tc_commit(bar(F_SFULL_A));
          }
          // PV_B(g)
          if (j == 0 && it > 0 && !mbar_wait(bar(F_OEMPTY_B), (it - 1) & 1, ctl, ERR_KERNEL_FWD + F_OEMPTY_B)) { ok = false; break; }
          if (!mbar_wait(bar(F_PFULL_B), gg & 1, ctl, ERR_KERNEL_FWD + F_PFULL_B)) { ok = false; break; }
          tc_fence_after();
          issue_pv(128, 256 + D, st, j == 0);
          tc_commit(bar(F_ODONE_B));
          tc_commit(bar(F_VEMPTY0 + st));
          // S_B(g+1)
          if (more) {
            const int st1 = (gg + 1) & 1;
            issue_s(sQB, 128, st1);
            tc_commit(bar(F_SFULL_B));
            tc_commit(bar(F_KEMPTY0 + st1));
            if (j + 2 == n) tc_commit(bar(F_QEMPTY));
          }
        }
        g0 += n;
      }
      tc_commit(bar(F_FINAL));
      mbar_drain(bar(F_FINAL), 0);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ RoPE warps
    const int rtid = tid - 256;
    uint32_t gk = 0, ntile = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++it) {
      int b, head, s, pair;
      decode_unit(g, n_pairs, u, b, head, s, pair);
      ok = mbar_wait(bar(F_QFULL), it & 1, ctl, ERR_KERNEL_FWD + F_QFULL);
      ok = rope_tile<D>(smem + Ly::QA_OFF, rowoff + (ntile++ & 1) * 128, 2 * pair * kTile, s, g, p.rope, tab, rtid, lane, ok);
      if (!ok) break;
      ok = rope_tile<D>(smem + Ly::QB_OFF, rowoff + (ntile++ & 1) * 128, (2 * pair + 1) * kTile, s, g, p.rope, tab, rtid,
                        lane, ok);
      if (!ok) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(F_QROT));
      for (int j = 0; j < g.n_tiles; ++j) {
        const uint32_t gg = gk + j;
        const int st = gg & 1;
        const uint32_t n = gg >> 1;
        ok = mbar_wait(bar(F_KFULL0 + st), n & 1, ctl, ERR_KERNEL_FWD + F_KFULL0 + st);
        ok = rope_tile<D>(smem + Ly::K_OFF + st * Ly::TILE, rowoff + (ntile++ & 1) * 128, j * kTile, s, g, p.rope,
                          tab, rtid, lane, ok);
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_KROT0 + st));
      }
      gk += g.n_tiles;
    }
  } else {
    // ------------------------------------------------------------ softmax warps (A: 0-3, B: 4-7)
    const int wg = warp >> 2;                              // 0 = Q tile A, 1 = Q tile B
    const int r = tid & 127;                               // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = wg ? 128u : 0u;
    const uint32_t colO = 256u + (wg ? (uint32_t)D : 0u);
    const int barS = wg ? F_SFULL_B : F_SFULL_A;
    const int barP = wg ? F_PFULL_B : F_PFULL_A;
    const int barO = wg ? F_ODONE_B : F_ODONE_A;
    const int barOE = wg ? F_OEMPTY_B : F_OEMPTY_A;
    const float sl2 = p.scale_log2;
    uint32_t g0 = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++it) {
      int b, head, s, pair;
      decode_unit(g, n_pairs, u, b, head, s, pair);
      const int tile = 2 * pair + wg;
      float m = 0.f, l = 0.f;
      for (int j = 0; j < g.n_tiles; ++j) {
        const uint32_t gg = g0 + j;
        if (!mbar_wait(bar(barS), gg & 1, ctl, ERR_KERNEL_FWD + barS)) { ok = false; break; }
        tc_fence_after();
        const int valid = min(kTile, g.L - j * kTile);
        // pass 1: row max (keys at or past `valid` only exist in the scope's last tile)
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (valid == kTile) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float x[32];
            tmem_ld32(tmem + lane_base + colS + c * 32, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], x[e]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float x[32];
            tmem_ld32(tmem + lane_base + colS + c * 32, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) m4[e & 3] = fmaxf(m4[e & 3], (c * 32 + e < valid) ? x[e] : -INFINITY);
          }
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
        if (j == 0) {
          m = mx;
        } else {
          const bool need = mx > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            // S_X(g) was issued after PV_X(g-1), so that P V is already complete;
            // the wait only orders this thread after it.
            if (!mbar_wait(bar(barO), (gg - 1) & 1, ctl, ERR_KERNEL_FWD + barO)) { ok = false; break; }
            tc_fence_after();
            const float m_new = need ? mx : m;
            const float f = ex2(m - m_new);
            m = m_new;
            l *= f;
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              float o[16];
              tmem_ld16(tmem + lane_base + colO + c * 16, o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] *= f;
              tmem_st16f(tmem + lane_base + colO + c * 16, o);
            }
            tmem_st_wait();
          }
        }
        // pass 2: P = 2^(S * scale * log2 e - m) as bf16 over the S columns already
        // read; the exponent argument and the row sum use packed two-lane fp32.
        const unsigned long long sl2x2 = f2_pack(sl2, sl2);
        const unsigned long long negm2 = f2_pack(-m, -m);
        unsigned long long acc2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float x[32];
          tmem_ld32(tmem + lane_base + colS + c * 32, x);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float t0, t1;
            f2_unpack(ffma2(f2_pack(x[2 * e], x[2 * e + 1]), sl2x2, negm2), t0, t1);
            float a = ex2(t0), bb = ex2(t1);
            if (valid < kTile) {
              a = (c * 32 + 2 * e < valid) ? a : 0.f;
              bb = (c * 32 + 2 * e + 1 < valid) ? bb : 0.f;
            }
            acc2[e & 1] = fadd2(acc2[e & 1], f2_pack(a, bb));
            pk[e] = pack_bf16(a, bb);
          }
          tmem_st16(tmem + lane_base + colS + c * 16, pk);
        }
        {
          float s0, s1, s2, s3;
          f2_unpack(acc2[0], s0, s1);
          f2_unpack(acc2[1], s2, s3);
          l += (s0 + s1) + (s2 + s3);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(barP));
      }
      if (!ok) break;
      // ---- epilogue: O / l to the token's original row, LSE in natural log.
      // S_X(glast) proved PV_X(glast-1) complete, so one parity wait suffices.
      const uint32_t glast = g0 + g.n_tiles - 1;
      if (!mbar_wait(bar(barO), glast & 1, ctl, ERR_KERNEL_FWD + barO)) break;
      tc_fence_after();
      const int prow = tile * kTile + r;
      const bool row_ok = prow < g.L;
      const int tok = row_ok ? token_of(g, s, prow) : 0;
      const float inv_l = 1.0f / l;
      uint16_t* orow = p.out + (((size_t)b * g.N + tok) * g.heads + head) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_base + colO + c * 32, o);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(o[8 * q4 + 0] * inv_l, o[8 * q4 + 1] * inv_l);
            w.y = pack_bf16(o[8 * q4 + 2] * inv_l, o[8 * q4 + 3] * inv_l);
            w.z = pack_bf16(o[8 * q4 + 4] * inv_l, o[8 * q4 + 5] * inv_l);
            w.w = pack_bf16(o[8 * q4 + 6] * inv_l, o[8 * q4 + 7] * inv_l);
            dst[q4] = w;
          }
        }
      }
      if (row_ok) p.lse[((size_t)b * g.heads + head) * g.N + tok] = (m + log2f(l)) * 0.6931471805599453f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(barOE));
      g0 += g.n_tiles;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t fwd_smem_bytes(int D, int rope_entries) {
  const size_t base = (D == 128) ? FwdLayout<128>::ROPE_OFF : FwdLayout<64>::ROPE_OFF;
  return base + (size_t)rope_entries * sizeof(float2);
}

int fwd_units(const Geom& g) { return g.B * g.heads * g.k * ((g.n_tiles + 1) / 2); }

cudaError_t launch_fwd(const FwdParams& p, int grid, cudaStream_t stream) {
  const size_t smem = fwd_smem_bytes(p.g.D, p.rope.entries);
  cudaError_t e;
  if (p.g.D == 128) {
    e = cudaFuncSetAttribute(skiparse_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    skiparse_fwd_kernel<128><<<grid, kFwdThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(skiparse_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    skiparse_fwd_kernel<64><<<grid, kFwdThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace skp
