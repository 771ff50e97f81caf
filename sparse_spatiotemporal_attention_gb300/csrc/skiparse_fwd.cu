// Skiparse attention forward: a RoPE pass and one persistent attention kernel.
//
// What it computes ("Open-Sora Plan" docs, "Skiparse Attention", single and
// group skip listings): for every (batch b, head, scope s) the softmax
// attention of the scope's L = N/k tokens among themselves, with q and k
// rotated by 3D RoPE at their original positions, written back to the tokens'
// original rows. The rearrange never happens in memory: the TMA tensor maps
// address the scope's rows directly (see skiparse_host.cu), and the epilogue
// stores each output row at its original token index.
//
// RoPE pass: one warp per (b, token, head) row rotates q and k once into the
// caller's workspace (row layout unchanged). Every K tile is read by all the
// query-tile pairs of its scope, so rotating it once here instead of in each
// attention CTA removes L/256 redundant rotations per tile.
//
// Attention: one work unit = (b, head, s, a pair of 128-row Q tiles A and B),
// so every K / V tile is loaded once for 256 query rows. Warp roles:
//   warps 0-3   softmax for Q tile A, one query row per thread (TMEM lane);
//   warps 4-7   softmax for Q tile B;
//   warp  8     TMA producer: rotated Q pair, then a 2-stage K / V ring;
//   warp  9     MMA issuer (tcgen05.mma kind::f16, fp32 accumulators in TMEM).
// The TMA and MMA warps run their loops with all lanes (waits voted across the
// warp), lane 0 issuing.
// TMEM columns: S_A / P_A 0..127, S_B / P_B 128..255, O_A 256.., O_B 384...
// MMA issue order: S_A(g), S_B(g), PV_A(g), S_A(g+1), PV_B(g), S_B(g+1), ...
// so each softmax warpgroup's critical loop is softmax + two MMA groups while
// the tensor core alternates between the two Q tiles. Because S_X(g) is issued
// after PV_X(g-1), the S-full barrier of tile g proves PV_X(g-1) complete, which
// keeps every parity wait on the O-done barriers one phase ahead at most.
// The softmax reads each 128-score row from TMEM in one load (row max, then
// exponentials from registers); online softmax with lazy O rescaling
// (threshold 2^8), P written back over S as bf16. The epilogue reads O in one
// load, releases its columns, then writes each out row (32-byte stores when
// out's base allows).
#include <type_traits>

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
  static constexpr int BYTES = V_OFF + 2 * TILE;
};

enum FwdBar {
  F_QFULL, F_QEMPTY,
  F_KFULL0, F_KFULL1, F_KEMPTY0, F_KEMPTY1,
  F_VFULL0, F_VFULL1, F_VEMPTY0, F_VEMPTY1,
  F_SFULL_A, F_SFULL_B, F_PFULL_A, F_PFULL_B, F_ODONE_A, F_ODONE_B, F_OEMPTY_A, F_OEMPTY_B, F_FINAL, F_NBARS
};

constexpr int kFwdThreads = 320;
constexpr int kPrefetchLead = 4;   // K tiles before an item's end at which the next item's Q pair is prefetched
constexpr int kRopeThreads = 256;

// P = 2^(S * sl2 - m) for one softmax row held in registers (x, 128 keys), as
// bf16 into TMEM at taddr (16 columns per 32 keys, over the row's S columns);
// returns the row sum of the unrounded P. The exponent argument and the sum use
// packed two-lane fp32. With RAGGED, keys at or past `valid` get P = 0.
template <bool RAGGED>
__device__ __forceinline__ float softmax_p_bf16(const float (&x)[kTile], uint32_t taddr, float sl2, float m,
                                                int valid) {
  const unsigned long long sl2x2 = f2_pack(sl2, sl2);
  const unsigned long long negm2 = f2_pack(-m, -m);
  unsigned long long acc2[2] = {0ull, 0ull};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int k0 = c * 32 + 2 * e;
      float t0, t1;
      f2_unpack(ffma2(f2_pack(x[k0], x[k0 + 1]), sl2x2, negm2), t0, t1);
      float a = ex2(t0), bb = ex2(t1);
      if constexpr (RAGGED) {
        a = k0 < valid ? a : 0.f;
        bb = k0 + 1 < valid ? bb : 0.f;
      }
      acc2[e & 1] = fadd2(acc2[e & 1], f2_pack(a, bb));
      pk[e] = pack_bf16(a, bb);
    }
    tmem_st16(taddr + c * 16, pk);
  }
  float s0, s1, s2, s3;
  f2_unpack(acc2[0], s0, s1);
  f2_unpack(acc2[1], s2, s3);
  return (s0 + s1) + (s2 + s3);
}

__device__ __forceinline__ void decode_unit(const Geom& g, int n_pairs, int u, int& b, int& head, int& s, int& pair) {
  pair = u % n_pairs;
  int r = u / n_pairs;
  s = g.s0 + (r % g.ks) * g.sstep;               // the ks scopes of this call
  r /= g.ks;
  head = r % g.heads;
  b = r / g.heads;
}

// Work item `it`: a whole unit, or one key-tile range [j0, j1) of a unit of the
// last round, split so that its pieces run on the SMs the round leaves idle
// (slot >= 0 indexes the piece's partial results). False when the item has no
// work: a Q-tile pair past a shorter scope's end, or an empty key range.
struct Item {
  int b, head, s, pair, nt, j0, j1, slot;
};

__device__ __forceinline__ bool decode_item(const FwdParams& p, int n_pairs, int it, Item& w) {
  int u = it, piece = 0;
  w.slot = -1;
  if (it >= p.n_full) {
    const int q = it - p.n_full;
    const int r = q / p.pieces;
    u = p.n_full + r;
    piece = q - r * p.pieces;
    w.slot = q;
  }
  decode_unit(p.g, n_pairs, u, w.b, w.head, w.s, w.pair);
  w.nt = scope_tiles(p.g, w.s);
  if (2 * w.pair >= w.nt) return false;             // a shorter scope has fewer Q-tile pairs
  if (w.slot < 0) {
    w.j0 = 0;
    w.j1 = w.nt;
  } else {
    w.j0 = piece * w.nt / p.pieces;
    w.j1 = (piece + 1) * w.nt / p.pieces;
  }
  return w.j1 > w.j0;
}

// ---------------------------------------------------------------------------
// RoPE pass: q, k (pre-RoPE) -> rotated copies in the workspace. One warp per
// (b, token, head) row, two rows per iteration so each lane has four 8-byte
// loads in flight; lane l owns channel pairs l*PPL .. l*PPL+PPL-1.
// ---------------------------------------------------------------------------
// The cos/sin table: one thread per entry, written to global memory once per call.
__global__ void __launch_bounds__(256) skiparse_rope_table_kernel(const RopeParams r, float2* tab) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < r.entries) {
    int pos;
    double om;
    rope_entry_args(r, e, pos, om);
    tab[e] = rope_cos_sin(pos, om);
  }
}

cudaError_t launch_rope_table(const RopeParams& r, float2* tab, cudaStream_t stream) {
  skiparse_rope_table_kernel<<<(r.entries + 255) / 256, 256, 0, stream>>>(r, tab);
  return cudaGetLastError();
}

template <int D>
__global__ void __launch_bounds__(kRopeThreads) skiparse_fwd_rope_kernel(const __grid_constant__ FwdParams p) {
  pdl_trigger();                                     // the attention kernel may take SMs as this pass drains
  extern __shared__ float2 tab[];
  const Geom& g = p.g;
  rope_load_table(tab, p.rope_gtab, p.rope.entries, threadIdx.x, blockDim.x);
  __syncthreads();
  constexpr int PPL = D / 64;
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  PairSel sel[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) sel[e] = pair_select(p.rope, lane * PPL + e);
  const long long rows = (long long)g.B * g.N * g.heads;
  const long long stride = (long long)gridDim.x * wpb;
  for (long long r0 = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); r0 < rows; r0 += 2 * stride) {
    uint32_t qv[2][PPL], kv[2][PPL];
    int tt[2], th[2], tw[2];
    bool skip[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long row = r0 + u * stride;
      skip[u] = row >= rows;
      if (skip[u]) continue;
      int b, i, head;
      row_coords(g, (int)row, b, i, head);
      if (g.ks < g.k) {                              // only the rows of the scopes this call computes
        int s, pos;
        scope_pos_of(g, i, s, pos);
        skip[u] = !in_subset(g, s);
        if (skip[u]) continue;
      }
      token_coords(p.rope, i, tt[u], th[u], tw[u]);
      const size_t base = (size_t)row * D + lane * 2 * PPL;
      if (PPL == 2) {
        const uint2 a = *reinterpret_cast<const uint2*>(p.q + base);
        const uint2 c = *reinterpret_cast<const uint2*>(p.k + base);
        qv[u][0] = a.x; qv[u][PPL - 1] = a.y; kv[u][0] = c.x; kv[u][PPL - 1] = c.y;
      } else {
        qv[u][0] = *reinterpret_cast<const uint32_t*>(p.q + base);
        kv[u][0] = *reinterpret_cast<const uint32_t*>(p.k + base);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long row = r0 + u * stride;
      if (skip[u]) continue;
      uint32_t qo[PPL], ko[PPL];
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        const float2 cs = tab[pair_index(sel[e], tt[u], th[u], tw[u])];
        const float2 a = rope_rotate(bf16lo(qv[u][e]), bf16hi(qv[u][e]), cs);
        const float2 c = rope_rotate(bf16lo(kv[u][e]), bf16hi(kv[u][e]), cs);
        qo[e] = pack_bf16(a.x, a.y);
        ko[e] = pack_bf16(c.x, c.y);
      }
      const size_t base = (size_t)row * D + lane * 2 * PPL;
      if (PPL == 2) {
        *reinterpret_cast<uint2*>(p.qr + base) = make_uint2(qo[0], qo[PPL - 1]);
        *reinterpret_cast<uint2*>(p.kr + base) = make_uint2(ko[0], ko[PPL - 1]);
      } else {
        *reinterpret_cast<uint32_t*>(p.qr + base) = qo[0];
        *reinterpret_cast<uint32_t*>(p.kr + base) = ko[0];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Pack pass (scopes of unequal length, N not divisible by k or k^2): q, k (rotated
// unless rope_theta = 0) and v gathered into scope order (k, B, Lp, heads, D),
// positions past each scope's end zero. One warp per scope-ordered row, two rows
// per iteration, head fastest so a warp's consecutive rows read one token's
// heads; lane l owns channel pairs l*PPL .. l*PPL+PPL-1.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kRopeThreads) skiparse_fwd_pack_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ float2 tab[];
  const Geom& g = p.g;
  if (p.rotate) rope_load_table(tab, p.rope_gtab, p.rope.entries, threadIdx.x, blockDim.x);
  __syncthreads();
  constexpr int PPL = D / 64;
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  PairSel sel[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) sel[e] = pair_select(p.rope, lane * PPL + e);
  const long long rows = (long long)g.k * g.B * g.Lp * g.heads;
  const long long stride = (long long)gridDim.x * wpb;
  for (long long r0 = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); r0 < rows; r0 += 2 * stride) {
    uint32_t qv[2][PPL], kv[2][PPL], vv[2][PPL];
    int tok[2];
    bool skip[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      tok[u] = -1;
      const long long row = r0 + u * stride;
      skip[u] = row >= rows;
      if (skip[u]) continue;
      const int sbp = fdiv((int)row, g.fheads);              // (s * B + b) * Lp + pos
      const int head = (int)row - sbp * g.heads;
      const int sb = fdiv(sbp, g.fLp);
      const int pos = sbp - sb * g.Lp;
      const int s = fdiv(sb, g.fB);
      const int b = sb - s * g.B;
      skip[u] = !in_subset(g, s);                    // the other scopes' rows are never read
      if (skip[u] || pos >= scope_len(g, s)) continue;
      tok[u] = token_of(g, s, pos);
      const size_t src = (((size_t)b * g.N + tok[u]) * g.heads + head) * D + lane * 2 * PPL;
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        qv[u][e] = *reinterpret_cast<const uint32_t*>(p.q + src + 2 * e);
        kv[u][e] = *reinterpret_cast<const uint32_t*>(p.k + src + 2 * e);
        vv[u][e] = *reinterpret_cast<const uint32_t*>(p.v + src + 2 * e);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long row = r0 + u * stride;
      if (skip[u]) continue;
      uint32_t qo[PPL], ko[PPL], vo[PPL];
#pragma unroll
      for (int e = 0; e < PPL; ++e) qo[e] = ko[e] = vo[e] = 0u;
      if (tok[u] >= 0) {
        int t = 0, hh = 0, w = 0;
        if (p.rotate) token_coords(p.rope, tok[u], t, hh, w);
#pragma unroll
        for (int e = 0; e < PPL; ++e) {
          vo[e] = vv[u][e];
          if (p.rotate) {
            const float2 cs = tab[pair_index(sel[e], t, hh, w)];
            const float2 a = rope_rotate(bf16lo(qv[u][e]), bf16hi(qv[u][e]), cs);
            const float2 c = rope_rotate(bf16lo(kv[u][e]), bf16hi(kv[u][e]), cs);
            qo[e] = pack_bf16(a.x, a.y);
            ko[e] = pack_bf16(c.x, c.y);
          } else {
            qo[e] = qv[u][e];
            ko[e] = kv[u][e];
          }
        }
      }
      const size_t dst = (size_t)row * D + lane * 2 * PPL;
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        *reinterpret_cast<uint32_t*>(p.qr + dst + 2 * e) = qo[e];
        *reinterpret_cast<uint32_t*>(p.kr + dst + 2 * e) = ko[e];
        *reinterpret_cast<uint32_t*>(p.vr + dst + 2 * e) = vo[e];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Attention over rotated q / k
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1) skiparse_fwd_kernel(const __grid_constant__ FwdParams p) {
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
  const uint32_t sQA = smem_u32(smem + Ly::QA_OFF);
  const uint32_t sQB = smem_u32(smem + Ly::QB_OFF);
  const uint32_t sK = smem_u32(smem + Ly::K_OFF);
  const uint32_t sV = smem_u32(smem + Ly::V_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const Ctl ctl{abort_flag, p.err};
  const Geom& g = p.g;
  const int n_pairs = (g.n_tiles + 1) >> 1;
  constexpr int E = ERR_KERNEL_FWD;

  if (tid == 0) {
    *abort_flag = 0;
    const uint32_t counts[F_NBARS] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 4, 4, 1, 1, 4, 4, 1};
    for (int i = 0; i < F_NBARS; ++i) mbar_init(bar(i), counts[i]);
    mbar_fence_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();                                        // the RoPE / pack pass's copies are complete
  auto warp_wait = [&](int i, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ctl, E + i)) != 0;
  };
  const bool leader = lane == 0;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (leader) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
    }
    uint32_t q_issued = 0, k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
    uint32_t gk = 0;
    int it = 0;
    bool ok = true;
    for (int wi = blockIdx.x; ok && wi < p.n_items; wi += gridDim.x) {
      Item w;
      if (!decode_item(p, n_pairs, wi, w)) continue;
      const int b = w.b, head = w.head, s = w.s, pair = w.pair;
      const int nt = w.j1 - w.j0;                    // K tiles of this item
      if (it > 0 && !warp_wait(F_QEMPTY, (it - 1) & 1)) break;
      if (leader) {
        mbar_expect_tx(bar(F_QFULL), 2 * Ly::TILE);
        const TileCoord tcA = scope_tile(g, s, b, 2 * pair * kTile);
        const TileCoord tcB = scope_tile(g, s, b, (2 * pair + 1) * kTile);
#pragma unroll
        for (int h = 0; h < Ly::HALVES; ++h) {
          load_tile(sQA + h * kHalfBytes, &p.tm_q, bar(F_QFULL), tcA, h * 64, head);
          load_tile(sQB + h * kHalfBytes, &p.tm_q, bar(F_QFULL), tcB, h * 64, head);
        }
      }
      __syncwarp();
      ++q_issued;
      // the next item's Q pair (read once, from HBM) is prefetched into L2 a few
      // K tiles before this item ends, so its load after QEMPTY hits L2
      Item wn;
      bool next = false;
      for (int wi2 = wi + gridDim.x; wi2 < p.n_items; wi2 += gridDim.x)
        if (decode_item(p, n_pairs, wi2, wn)) {
          next = true;
          break;
        }
      const int pf_at = nt > kPrefetchLead ? nt - kPrefetchLead : 0;
      for (int jj = 0; jj < nt; ++jj) {
        const int j = w.j0 + jj;                     // the scope's K tile
        const uint32_t gg = gk + jj;
        const int st = gg & 1;
        const uint32_t n = gg >> 1;
        const TileCoord tcj = scope_tile(g, s, b, j * kTile);
        if (leader && next && jj == pf_at) {
          const TileCoord nA = scope_tile(g, wn.s, wn.b, 2 * wn.pair * kTile);
          const TileCoord nB = scope_tile(g, wn.s, wn.b, (2 * wn.pair + 1) * kTile);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h) {
            prefetch_tile(&p.tm_q, nA, h * 64, wn.head);
            prefetch_tile(&p.tm_q, nB, h * 64, wn.head);
          }
        }
        if (n > 0 && !warp_wait(F_KEMPTY0 + st, (n - 1) & 1)) { ok = false; break; }
        if (leader) {
          mbar_expect_tx(bar(F_KFULL0 + st), Ly::TILE);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            load_tile(sK + st * Ly::TILE + h * kHalfBytes, &p.tm_k, bar(F_KFULL0 + st), tcj, h * 64, head);
        }
        __syncwarp();
        ++k_issued[st];
        if (n > 0 && !warp_wait(F_VEMPTY0 + st, (n - 1) & 1)) { ok = false; break; }
        if (leader) {
          mbar_expect_tx(bar(F_VFULL0 + st), Ly::TILE);
#pragma unroll
          for (int h = 0; h < Ly::HALVES; ++h)
            load_tile(sV + st * Ly::TILE + h * kHalfBytes, &p.tm_v, bar(F_VFULL0 + st), tcj, h * 64, head);
        }
        __syncwarp();
        ++v_issued[st];
      }
      gk += nt;
      ++it;
    }
    // Copies still in flight (only after an abort) must land before exit.
    if (leader) {
      if (q_issued) mbar_drain(bar(F_QFULL), (q_issued - 1) & 1);
      for (int st = 0; st < 2; ++st) {
        if (k_issued[st]) mbar_drain(bar(F_KFULL0 + st), (k_issued[st] - 1) & 1);
        if (v_issued[st]) mbar_drain(bar(F_VFULL0 + st), (v_issued[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 alone issues while the other lanes wait at the warp's final sync.
    // Its waits nearly always find the barrier complete, and a wait without
    // the warp vote and reconvergence costs the issuing thread (which, not the
    // tensor core, sets this kernel's pace) fewer cycles.
    if (leader) {
      auto lane_wait = [&](int i, uint32_t parity) -> bool { return mbar_wait(bar(i), parity, ctl, E + i); };
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
      uint32_t g0 = 0;
      int it = 0;
      bool ok = true;
      // operand descriptors of k-step 0, per tile and stage (k-steps add a constant)
      const uint64_t dQA = desc_kmajor(sQA, 0), dQB = desc_kmajor(sQB, 0);
      const uint64_t dK0 = desc_kmajor(sK, 0), dK1 = desc_kmajor(sK + Ly::TILE, 0);
      const uint64_t dV0 = desc_mnmajor(sV, 0), dV1 = desc_mnmajor(sV + Ly::TILE, 0);
      // S_X = Q_X K_g^T into TMEM columns colS (X = A: 0, B: 128)
      auto issue_s = [&](uint64_t dq, uint32_t colS, int st) {
        const uint64_t dk = st ? dK1 : dK0;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + colS, kmajor_step(dq, ks), kmajor_step(dk, ks), kIdS, ks > 0 ? 1u : 0u);
      };
      // O_X += P_X V_g, P_X in TMEM over S_X
      auto issue_pv = [&](uint32_t colS, uint32_t colO, int st, bool first) {
        const uint64_t dv = st ? dV1 : dV0;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ts(tmem + colO, tmem + colS + ks * 8, mnmajor_step(dv, ks), kIdPV, (!first || ks > 0) ? 1u : 0u);
      };
      for (int wi = blockIdx.x; ok && wi < p.n_items; wi += gridDim.x) {
        Item w;
        if (!decode_item(p, n_pairs, wi, w)) continue;
        const int n = w.j1 - w.j0;                   // K tiles of this item
        if (!lane_wait(F_QFULL, it & 1)) break;
        if (!lane_wait(F_KFULL0 + (g0 & 1), (g0 >> 1) & 1)) break;
        tc_fence_after();
        issue_s(dQA, 0, g0 & 1);
        tc_commit(bar(F_SFULL_A));
        issue_s(dQB, 128, g0 & 1);
        tc_commit(bar(F_SFULL_B));
        tc_commit(bar(F_KEMPTY0 + (g0 & 1)));
        if (n == 1) tc_commit(bar(F_QEMPTY));
        for (int j = 0; j < n; ++j) {
          const uint32_t gg = g0 + j;
          const int st = gg & 1;
          const uint32_t nn = gg >> 1;
          // PV_A(g)
          if (j == 0 && it > 0 && !lane_wait(F_OEMPTY_A, (it - 1) & 1)) { ok = false; break; }
          if (!lane_wait(F_PFULL_A, gg & 1)) { ok = false; break; }
          if (!lane_wait(F_VFULL0 + st, nn & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, 256, st, j == 0);
          tc_commit(bar(F_ODONE_A));
          // S_A(g+1)
          const bool more = j + 1 < n;
          const int st1 = (gg + 1) & 1;
          if (more) {
            if (!lane_wait(F_KFULL0 + st1, ((gg + 1) >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_s(dQA, 0, st1);
            tc_commit(bar(F_SFULL_A));
          }
          // PV_B(g)
          if (j == 0 && it > 0 && !lane_wait(F_OEMPTY_B, (it - 1) & 1)) { ok = false; break; }
          if (!lane_wait(F_PFULL_B, gg & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(128, 256 + D, st, j == 0);
          tc_commit(bar(F_ODONE_B));
          tc_commit(bar(F_VEMPTY0 + st));
          // S_B(g+1)
          if (more) {
            issue_s(dQB, 128, st1);
            tc_commit(bar(F_SFULL_B));
            tc_commit(bar(F_KEMPTY0 + st1));
            if (j + 2 == n) tc_commit(bar(F_QEMPTY));
          }
        }
        g0 += n;
        ++it;
      }
      tc_commit(bar(F_FINAL));
      mbar_drain(bar(F_FINAL), 0);
    }
    __syncwarp();
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
    for (int wi = blockIdx.x; ok && wi < p.n_items; wi += gridDim.x) {
      Item w;
      if (!decode_item(p, n_pairs, wi, w)) continue;
      const int b = w.b, head = w.head, s = w.s, pair = w.pair;
      const int nt = w.j1 - w.j0;                    // K tiles of this item
      const int Ls = scope_len(g, s);
      const int tile = 2 * pair + wg;
      float m = 0.f, l = 0.f;
      for (int jj = 0; jj < nt; ++jj) {
        const int j = w.j0 + jj;                     // the scope's K tile
        const uint32_t gg = g0 + jj;
        if (!mbar_wait(bar(barS), gg & 1, ctl, ERR_KERNEL_FWD + barS)) { ok = false; break; }
        tc_fence_after();
        const int valid = min(kTile, Ls - j * kTile);
        // the whole S row in registers with one TMEM round trip
        float x[kTile];
        tmem_ld128(tmem + lane_base + colS, x);
        const float mx = (valid == kTile ? row_max128<false>(x, valid) : row_max128<true>(x, valid)) * sl2;
        float f = 1.f;
        bool rescale = false;
        if (jj == 0) {
          m = mx;
        } else {
          const bool need = mx > m + 8.0f;
          rescale = __any_sync(0xffffffffu, need);
          if (rescale) {
            const float m_new = need ? mx : m;
            f = ex2(m - m_new);
            m = m_new;
            l *= f;
          }
        }
        // P over the S columns (the full-tile path has no masking)
        l += valid == kTile ? softmax_p_bf16<false>(x, tmem + lane_base + colS, sl2, m, valid)
                            : softmax_p_bf16<true>(x, tmem + lane_base + colS, sl2, m, valid);
        if (rescale) {
          // O *= 2^(m_old - m_new) before P V adds this tile. S_X(g) was issued
          // after PV_X(g-1), so that P V is already complete; the wait only
          // orders this thread after it.
          if (!mbar_wait(bar(barO), (gg - 1) & 1, ctl, ERR_KERNEL_FWD + barO)) {
            tmem_st_wait();
            ok = false;
            break;
          }
          tc_fence_after();
          if constexpr (D == 128) {
            float o[128];
            tmem_ld128(tmem + lane_base + colO, o);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float oc[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) oc[e] = o[c * 16 + e] * f;
              tmem_st16f(tmem + lane_base + colO + c * 16, oc);
            }
          } else {
            float o[64];
            tmem_ld64(tmem + lane_base + colO, o);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float oc[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) oc[e] = o[c * 16 + e] * f;
              tmem_st16f(tmem + lane_base + colO + c * 16, oc);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(barP));
      }
      if (!ok) break;
      // ---- epilogue: O / l to the token's original row, LSE in natural log.
      // S_X(glast) proved PV_X(glast-1) complete, so one parity wait suffices.
      const uint32_t glast = g0 + nt - 1;
      if (!mbar_wait(bar(barO), glast & 1, ctl, ERR_KERNEL_FWD + barO)) break;
      tc_fence_after();
      const int prow = tile * kTile + r;
      if (w.slot >= 0) {
        // a piece of a split unit: unnormalised O and (m, l) for the merge
        float* po = p.part_o + ((size_t)w.slot * 256 + wg * kTile + r) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + colO + c * 32, o);
          float4* dst = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
        }
        p.part_ml[(size_t)w.slot * 256 + wg * kTile + r] = make_float2(m, l);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(barOE));
        g0 += nt;
        ++it;
        continue;
      }
      const bool row_ok = prow < Ls;
      const int tok = row_ok ? token_of(g, s, prow) : 0;
      const float inv_l = 1.0f / l;
      // the whole O row out of TMEM in one round trip, normalised and packed;
      // the O columns are released before the global stores, so the next
      // unit's first P V does not wait for them
      uint32_t pk[D / 2];
      {
        float o[D];
        if constexpr (D == 128) tmem_ld128(tmem + lane_base + colO, o);
        else tmem_ld64(tmem + lane_base + colO, o);
#pragma unroll
        for (int e = 0; e < D / 2; ++e) pk[e] = pack_bf16(o[2 * e] * inv_l, o[2 * e + 1] * inv_l);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(barOE));
      if (row_ok) {
        uint16_t* orow = p.out + (((size_t)b * g.N + tok) * g.heads + head) * D;
        // 32-byte stores when out's base allows them (rows are D * 2 bytes apart)
        if ((reinterpret_cast<uintptr_t>(p.out) & 31u) == 0) {
#pragma unroll
          for (int q8 = 0; q8 < D / 16; ++q8)
            st_global_32b(orow + 16 * q8, pk[8 * q8], pk[8 * q8 + 1], pk[8 * q8 + 2], pk[8 * q8 + 3], pk[8 * q8 + 4],
                          pk[8 * q8 + 5], pk[8 * q8 + 6], pk[8 * q8 + 7]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int q4 = 0; q4 < D / 8; ++q4) dst[q4] = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
        p.lse[((size_t)b * g.heads + head) * g.N + tok] = (m + log2f(l)) * 0.6931471805599453f;
      }
      g0 += nt;
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Merge of split units: one warp per row of a split unit's Q-tile pair. The
// pieces' partial results (O unnormalised, row max m and sum l, base 2) combine
// as O = sum_p 2^(m_p - M) O_p / L with M = max_p m_p and L = sum_p 2^(m_p - M) l_p,
// LSE = (M + log2 L) ln 2; out and lse are written at the token's row.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) skiparse_fwd_merge_kernel(const __grid_constant__ FwdParams p) {
  pdl_wait();                                        // the attention kernel's partials are complete
  const Geom& g = p.g;
  constexpr int CPL = D / 32;                        // channels per lane
  const int lane = threadIdx.x & 31;
  const int n_pairs = (g.n_tiles + 1) >> 1;
  const int np = p.pieces;
  const int units = (p.n_items - p.n_full) / np;
  const int rows = units * 256;
  for (int rr = blockIdx.x * 8 + (threadIdx.x >> 5); rr < rows; rr += gridDim.x * 8) {
    const int r = rr >> 8, row = rr & 255;
    int b, head, s, pair;
    decode_unit(g, n_pairs, p.n_full + r, b, head, s, pair);
    const int nt = scope_tiles(g, s);
    if (2 * pair >= nt) continue;
    const int prow = (2 * pair + (row >> 7)) * kTile + (row & 127);
    if (prow >= scope_len(g, s)) continue;
    const float2* ml = p.part_ml + (size_t)r * np * 256 + row;     // piece pc at ml[pc * 256]
    // the row's largest m over the pieces, lanes striding the pieces (an empty
    // key range wrote nothing and weighs 0)
    float M = -INFINITY;
    for (int pc = lane; pc < np; pc += 32)
      if ((pc + 1) * nt / np > pc * nt / np) M = fmaxf(M, ml[(size_t)pc * 256].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    // O and l: all pieces' loads issued ahead of their sums
    float L = 0.f, acc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = 0.f;
    const float* po = p.part_o + ((size_t)r * np * 256 + row) * D + lane * CPL;
    // a lane's CPL channels of a piece in one vector load (16 or 8 bytes)
    using VecT = typename std::conditional<CPL == 4, float4, float2>::type;
#pragma unroll 16
    for (int pc = 0; pc < np; ++pc) {
      const float2 v = ml[(size_t)pc * 256];
      const bool has = (pc + 1) * nt / np > pc * nt / np;
      const float f = has ? ex2(v.x - M) : 0.f;
      L = fmaf(f, has ? v.y : 0.f, L);
      const VecT q = *reinterpret_cast<const VecT*>(po + (size_t)pc * 256 * D);
      const float* qe = reinterpret_cast<const float*>(&q);
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc[e] = fmaf(f, has ? qe[e] : 0.f, acc[e]);
    }
    const int tok = token_of(g, s, prow);
    const float inv = 1.0f / L;
    uint16_t* orow = p.out + (((size_t)b * g.N + tok) * g.heads + head) * D + lane * CPL;
#pragma unroll
    for (int e = 0; e < CPL; e += 2) *reinterpret_cast<uint32_t*>(orow + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0) p.lse[((size_t)b * g.heads + head) * g.N + tok] = (M + log2f(L)) * 0.6931471805599453f;
  }
}

cudaError_t launch_fwd_merge(const FwdParams& p, int sms, cudaStream_t stream) {
  const int rows = (p.n_items - p.n_full) / p.pieces * 256;
  int grid = (rows + 7) / 8;
  if (grid > 4 * sms) grid = 4 * sms;
  if (p.g.D == 128) return launch_after_previous(skiparse_fwd_merge_kernel<128>, grid, 256, 0, stream, p);
  return launch_after_previous(skiparse_fwd_merge_kernel<64>, grid, 256, 0, stream, p);
}

size_t fwd_smem_bytes(int D) { return D == 128 ? FwdLayout<128>::BYTES : FwdLayout<64>::BYTES; }

size_t fwd_rope_smem_bytes(int rope_entries) { return (size_t)rope_entries * sizeof(float2); }

int fwd_units(const Geom& g) { return g.B * g.heads * g.ks * ((g.n_tiles + 1) / 2); }

cudaError_t launch_fwd_rope(const FwdParams& p, int grid, int sms, cudaStream_t stream) {
  const size_t smem = fwd_rope_smem_bytes(p.rope.entries);
  cudaError_t e;
  if (p.g.D == 128) {
    e = cudaFuncSetAttribute(skiparse_fwd_rope_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    grid = one_wave(skiparse_fwd_rope_kernel<128>, grid, kRopeThreads, smem, sms);
    skiparse_fwd_rope_kernel<128><<<grid, kRopeThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(skiparse_fwd_rope_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    grid = one_wave(skiparse_fwd_rope_kernel<64>, grid, kRopeThreads, smem, sms);
    skiparse_fwd_rope_kernel<64><<<grid, kRopeThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd_pack(const FwdParams& p, int grid, int sms, cudaStream_t stream) {
  const size_t smem = p.rotate ? fwd_rope_smem_bytes(p.rope.entries) : 0;
  cudaError_t e;
  if (p.g.D == 128) {
    e = cudaFuncSetAttribute(skiparse_fwd_pack_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    grid = one_wave(skiparse_fwd_pack_kernel<128>, grid, kRopeThreads, smem, sms);
    skiparse_fwd_pack_kernel<128><<<grid, kRopeThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(skiparse_fwd_pack_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    grid = one_wave(skiparse_fwd_pack_kernel<64>, grid, kRopeThreads, smem, sms);
    skiparse_fwd_pack_kernel<64><<<grid, kRopeThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, int grid, cudaStream_t stream) {
  const size_t smem = fwd_smem_bytes(p.g.D);
  cudaError_t e;
  if (p.g.D == 128) {
    e = cudaFuncSetAttribute(skiparse_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_after_previous(skiparse_fwd_kernel<128>, grid, kFwdThreads, smem, stream, p);
  }
  e = cudaFuncSetAttribute(skiparse_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_after_previous(skiparse_fwd_kernel<64>, grid, kFwdThreads, smem, stream, p);
}

}  // namespace skp
