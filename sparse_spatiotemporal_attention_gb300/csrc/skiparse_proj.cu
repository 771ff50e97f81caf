// Q/K/V projection with the RoPE epilogue: the step before the attention in
// Open-Sora Plan's Skiparse listings ("Open-Sora Plan" docs, "Skiparse
// Attention", single- and group-skip implementations: q, k, v = Q(x), K(x),
// V(x), then RoPE on q and k at each token's original position).
//
//   [q | k | v] = x W^T (+ bias)       x (B N, C) bf16, W (3 heads D, C) bf16
//   q, k <- RoPE(t, h, w) in fp32 on the accumulator, one bf16 rounding
//
// skiparse_qkv_rope_kernel<BN>: persistent CTA pairs (clusters of two, one
// CTA per SM); a pair computes a 256-row x BN-column output tile with 2-SM
// MMAs (cta_group::2, M = 256: each CTA's 128 rows land in its own TMEM).
// Per CTA, 6 warps:
//   warp 0      TMA producer: 64-channel stages of the CTA's 128-row x tile
//               and its half (BN/2 rows) of the W tile, 128 channels per
//               stage as two 128-byte swizzled boxes, 3 stages of 64 KB;
//   warp 1      CTA 0: MMA issuer (converged, lane 0 issues 4 pair MMAs
//               M=256 N=BN K=16 per stage into one of two accumulators);
//               both CTAs' copies of a stage complete on CTA 0's barrier;
//   warps 2-5   epilogue: each thread one output row (its TMEM lane); bias,
//               RoPE from the shared-memory cos/sin table for the q and k
//               column ranges, bf16, stores into (B, N, heads, D).
// Two accumulators of BN columns let a tile's epilogue overlap the next
// tile's main loop. A stage costs each SM 32 KB of L2 reads per 512 tensor
// cycles (half of W per CTA), and one thread issues the MMAs of two SMs. Tile
// pairs run n-block fastest, so a wave shares a few x row blocks (read from
// HBM once) while W stays in L2.
#include "skiparse_internal.h"

namespace skp {

namespace {

constexpr int kProjThreads = 192;
constexpr int kPBM = 128;                 // output rows per tile
constexpr int kPBK = 64;                  // channels per box (one 128-byte row of bf16)
constexpr int kBoxes = 2;                 // boxes per stage: 128 channels, 8 MMA k-steps per wait
constexpr int kABox = kPBM * kPBK * 2;    // 16 KB
constexpr int kABytes = kBoxes * kABox;   // 32 KB
constexpr int kMaxStages = 6;

// barrier indices
enum : int {
  P_FULL0 = 0,                       // .. +5: stage landed in both CTAs (CTA 0's barrier)
  P_EMPTY0 = 6,                      // .. +5: stage consumed (pair MMA commit, both CTAs)
  P_ACCF0 = 12,                      // .. +1: accumulator ready (pair MMA commit, both CTAs)
  P_ACCE0 = 14,                      // .. +1: accumulator drained (CTA 0: 4 epilogue warps of each CTA)
  P_FINAL = 16,                      // every MMA done (teardown, CTA 0)
  P_NBARS = 17,
};

// The RoPE table with positions innermost: entry (axis, pair j, pos) at
// base(axis) + j * npos(axis) + pos, so the 32 rows of an epilogue warp (32
// consecutive tokens, usually consecutive w) read consecutive words. Same
// values as rope_build_table (rope_cos_sin).
__device__ __forceinline__ void proj_build_table(float2* tab, const RopeParams& r, int tid, int nthreads) {
  const int nt = r.T * r.dt2, nh = r.H * r.dh2;
  for (int e = tid; e < r.entries; e += nthreads) {
    int pos, j, dst;
    double om;
    if (e < nt) {
      pos = e / r.dt2; j = e - pos * r.dt2; om = r.om_t[j]; dst = j * r.T + pos;
    } else if (e < nt + nh) {
      const int e2 = e - nt; pos = e2 / r.dh2; j = e2 - pos * r.dh2; om = r.om_hw[j]; dst = nt + j * r.H + pos;
    } else {
      const int e2 = e - nt - nh; pos = e2 / r.dh2; j = e2 - pos * r.dh2; om = r.om_hw[j];
      dst = nt + nh + j * r.W + pos;
    }
    tab[dst] = rope_cos_sin(pos, om);
  }
}

// (cos, sin) of channel pair pp (0 .. D/2-1) at (t, h, w) in the table above
__device__ __forceinline__ float2 proj_cs(const float2* tab, const RopeParams& r, int pp, int t, int h, int w) {
  const int nt = r.T * r.dt2, nh = r.H * r.dh2;
  if (pp < r.dt2) return tab[pp * r.T + t];
  if (pp < r.dt2 + r.dh2) return tab[nt + (pp - r.dt2) * r.H + h];
  return tab[nt + nh + (pp - r.dt2 - r.dh2) * r.W + w];
}

}  // namespace

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kProjThreads, 1)
    skiparse_qkv_rope_kernel(const __grid_constant__ ProjParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kBBox = BN / 2 * kPBK * 2;                 // this CTA's half of the W tile, one box
  constexpr int kBBytes = kBoxes * kBBox;
  constexpr int kStage = kABytes + kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  int* abort_flag = reinterpret_cast<int*>(smem + 264);
  float2* tab = reinterpret_cast<float2*>(smem + 1024);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const uint32_t st0 = smem_u32(smem) + (uint32_t)p.stage_off;
  if ((st0 & 1023u) != 0 || p.stages < 2 || p.stages > kMaxStages) {   // swizzled stages: 1024-byte alignment
    if (tid == 0) atomicCAS(p.err, 0, ERR_SMEM_ALIGN);
    return;
  }
  const Ctl ctl{abort_flag, p.err};
  constexpr int E = ERR_KERNEL_PROJ;
  const int stages = p.stages;
  const int rank = (int)cluster_ctarank();
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_total = ((p.m_tiles + 1) >> 1) * p.n_tiles;     // 256-row tile pairs
  constexpr uint16_t kBoth = 3;

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < P_NBARS; ++i) {
      uint32_t cnt = 1;
      if (i == P_ACCE0 || i == P_ACCE0 + 1) cnt = 8;                        // epilogue warps of both CTAs
      mbar_init(bar(i), cnt);
    }
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), 2 * BN);   // the same columns in both SMs
  proj_build_table(tab, p.rope, tid, kProjThreads);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();        // both CTAs' barriers exist before any multicast targets them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto warp_wait = [&](int i, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ctl, E + i)) != 0;
  };
  // for barriers that also receive arrivals from the other CTA
  auto warp_wait_cl = [&](int i, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait_cl(bar(i), parity, ctl, E + i)) != 0;
  };
  const bool leader = lane == 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (leader) {
      tma_prefetch_map(&p.tm_x);
      tma_prefetch_map(&p.tm_w);
    }
    uint32_t it = 0;
    bool ok = true;
    for (int t = cid; ok && t < n_total; t += n_clusters) {
      const int nb = t % p.n_tiles, mb = 2 * (t / p.n_tiles) + rank;   // mb may be past the rows: zero fill
      for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
        const int s = (int)(it % (uint32_t)stages);
        const uint32_t use = it / (uint32_t)stages;
        if (use > 0 && !warp_wait_cl(P_EMPTY0 + s, (use - 1) & 1)) { ok = false; break; }
        if (leader) {
          // own x tile and own half of the W tile, both completing on CTA 0's barrier
          const uint32_t a = st0 + (uint32_t)(s * kStage);
          const uint32_t full = mapa_shared(bar(P_FULL0 + s), 0);
          if (rank == 0) mbar_expect_tx(bar(P_FULL0 + s), 2 * kStage);
#pragma unroll
          for (int h = 0; h < kBoxes; ++h) {
            const int c0 = (ks * kBoxes + h) * kPBK;        // past C: the box fills with zeros
            tma_load_2d_pair(a + h * kABox, &p.tm_x, full, c0, mb * kPBM);
            tma_load_2d_pair(a + kABytes + h * kBBox, &p.tm_w, full, c0, nb * BN + rank * (BN / 2));
          }
        }
        __syncwarp();
      }
    }
    // copies into this CTA land, and the pair MMAs' commits for every stage
    // arrive, before the pair may release its shared memory
    if (leader) {
      for (int s = 0; s < stages; ++s) {
        const uint32_t issued = it > (uint32_t)s ? (it - 1 - (uint32_t)s) / (uint32_t)stages + 1 : 0;
        if (issued) {
          if (rank == 0) mbar_drain_cl(bar(P_FULL0 + s), (issued - 1) & 1);   // both CTAs' copies
          mbar_drain_cl(bar(P_EMPTY0 + s), (issued - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && rank == 0) {
    // ------------------------------------------------------------ CTA 0: MMA issuer for the pair
    constexpr uint32_t kId = idesc_bf16(2 * kPBM, BN, false, false);
    uint32_t it = 0;
    int tl = 0;
    bool ok = true;
    for (int t = cid; ok && t < n_total; t += n_clusters, ++tl) {
      const int a = tl & 1;
      const uint32_t use = (uint32_t)tl >> 1;
      if (use > 0 && !warp_wait_cl(P_ACCE0 + a, (use - 1) & 1)) break;
      tc_fence_after();
      const uint32_t dacc = tmem + (uint32_t)(a * BN);
      for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
        const int s = (int)(it % (uint32_t)stages);
        if (!warp_wait_cl(P_FULL0 + s, (it / (uint32_t)stages) & 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          const uint32_t sa = st0 + (uint32_t)(s * kStage);
          const uint64_t da = desc_kmajor(sa, 0), db = desc_kmajor(sa + kABytes, 0);
#pragma unroll
          for (int kk = 0; kk < kBoxes * kPBK / 16; ++kk)
            mma_pair_ss(dacc, kmajor_step(da, kk, kABox), kmajor_step(db, kk, kBBox), kId, (ks > 0 || kk > 0) ? 1u : 0u);
          tc_commit_pair_mc(bar(P_EMPTY0 + s), kBoth);        // the stage is free in both CTAs
          if (ks + 1 == p.k_steps) tc_commit_pair_mc(bar(P_ACCF0 + a), kBoth);
        }
        __syncwarp();
      }
    }
    if (leader) {
      tc_commit_pair_mc(bar(P_FINAL), 1);
      mbar_drain_cl(bar(P_FINAL), 0);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue warps 2-5
    const int quarter = warp & 3;                          // TMEM lanes 32 quarter .. +31
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int tl = 0;
    for (int t = cid; t < n_total; t += n_clusters, ++tl) {
      const int a = tl & 1;
      if (!mbar_wait_cl(bar(P_ACCF0 + a), ((uint32_t)tl >> 1) & 1, ctl, E + P_ACCF0 + a)) break;
      tc_fence_after();
      const int nb = t % p.n_tiles, mb = 2 * (t / p.n_tiles) + rank;
      const int row = mb * kPBM + quarter * 32 + lane;     // b N + token
      const bool row_ok = row < p.M;
      const int n0 = nb * BN;                              // column in [q | k | v]
      const int region = n0 / p.hd;                        // 0 q, 1 k, 2 v (BN divides heads D)
      const int col0 = n0 - region * p.hd;                 // column in (heads, D)
      uint16_t* dst = region == 0 ? p.q : (region == 1 ? p.k : p.v);
      int tt = 0, hh = 0, ww = 0;
      if (row_ok && region < 2) {
        const int tok = row - fdiv(row, p.fN) * p.fN.d;
        token_coords(p.rope, tok, tt, hh, ww);
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float x[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(a * BN + c * 32), x);
        if (p.bias) {
          const uint4* bp = reinterpret_cast<const uint4*>(p.bias + n0 + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 u = __ldg(bp + q4);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              x[8 * q4 + 2 * e] += bf16lo(w4[e]);
              x[8 * q4 + 2 * e + 1] += bf16hi(w4[e]);
            }
          }
        }
        if (region < 2) {
          const int d0 = (col0 + c * 32) % p.D;            // channel of x[0] within its head
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 cs = proj_cs(tab, p.rope, d0 / 2 + e, tt, hh, ww);
            const float2 r = rope_rotate(x[2 * e], x[2 * e + 1], cs);
            x[2 * e] = r.x;
            x[2 * e + 1] = r.y;
          }
        }
        if (row_ok) {
          uint4* o = reinterpret_cast<uint4*>(dst + (size_t)row * p.hd + col0 + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(x[8 * q4 + 0], x[8 * q4 + 1]);
            w.y = pack_bf16(x[8 * q4 + 2], x[8 * q4 + 3]);
            w.z = pack_bf16(x[8 * q4 + 4], x[8 * q4 + 5]);
            w.w = pack_bf16(x[8 * q4 + 6], x[8 * q4 + 7]);
            o[q4] = w;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (leader) {
        if (rank == 0) mbar_arrive(bar(P_ACCE0 + a));
        else mbar_arrive_remote(mapa_shared(bar(P_ACCE0 + a), 0));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();        // neither CTA leaves, or frees the pair's TMEM, while the other may use it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * BN);
  }
}

int proj_bn(int hd) { return hd % 256 == 0 ? 256 : 128; }

size_t proj_stage_bytes(int bn) { return (size_t)kABytes + (size_t)kBoxes * (bn / 2) * kPBK * 2; }

int proj_stage_channels() { return kBoxes * kPBK; }

// barriers and flags (1 KB), then the RoPE table, rounded up to 1 KB
size_t proj_header_bytes(int rope_entries) { return 1024 + (((size_t)rope_entries * 8 + 1023) & ~(size_t)1023); }

namespace {

// Launch with at most as many CTA pairs as can be resident at once (an SM
// left over in a GPC cannot host half a pair).
template <class K>
cudaError_t launch_pairs(K kernel, const ProjParams& p, int grid, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kProjThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess && clusters > 0 && 2 * clusters < grid)
    grid = 2 * clusters;
  cudaGetLastError();
  kernel<<<grid, kProjThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_proj(const ProjParams& p, int bn, int grid, cudaStream_t stream) {
  const size_t smem = (size_t)p.stage_off + (size_t)p.stages * proj_stage_bytes(bn);
  if (bn == 256) return launch_pairs(skiparse_qkv_rope_kernel<256>, p, grid, smem, stream);
  return launch_pairs(skiparse_qkv_rope_kernel<128>, p, grid, smem, stream);
}

}  // namespace skp
