// Skiparse attention forward with 8-bit operands: the Wan 2.1 report, section 4
// "Model Design and Acceleration", 4.4.3 "Quantization", paragraph "8-Bit
// FlashAttention" (8-bit operands for S = Q K^T and O = P V, fp32 accumulation
// across key blocks), applied to the Skiparse forward pass of "Open-Sora Plan"
// docs, "Skiparse Attention". D = 128.
//
// Two recipes share these kernels (template parameter SI8):
//   * SI8 = true, the page's "Mixed 8-Bit optimization": INT8 q and k for
//     S = Q K^T, E4M3 P and v for O = P V. sm_103a has no 8-bit integer MMA
//     (ptxas: ".kind::i8 not supported on .target 'sm_103a'"), so the INT8
//     codes are stored as bf16 values (every integer up to 256 is exact in
//     bf16) and S runs as a kind::f16 MMA: every product is an integer below
//     2^14 and every partial sum of a 128-channel row an integer below 2^21,
//     all exact in the fp32 accumulator, so S is the exact INT8 dot product;
//   * SI8 = false, FlashAttention-3's native FP8: E4M3 q, k, v and P
//     (kind::f8f6f4 for both products), the recipe the page improves on.
// Quantization (readings; the page gives the recipe for Hopper): q after RoPE
// per (token, head) row, k after RoPE per block of 128 consecutive keys of a
// scope (one scale per K tile), v per (batch, head, channel) over all tokens;
// scale = max|x| / Q, codes RNE(x * Q / max|x|), Q = 127 (INT8) or 448 (E4M3).
// P relative to an integer base-2 row reference M enters O = P V as
// E4M3(2^8 P); O accumulates in fp32 TMEM across K tiles (the tensor memory
// accumulator is fp32, which is what the page's "FP32 accumulation for
// cross-block reduction" asks of the Hopper register path). The kernel keeps
// an integer reference m <= M (raised to the ceiling of a K tile's row max only
// when that exceeds m by more than 2) and quantizes 2^6 * 2^(t - m), which is
// E4M3(2^8 P) times the exact power of two 2^(M - m - 2): the same codes in
// E4M3's normal range, never above 256 < 448.
//
// Kernels:
//   skiparse_fwd8_vmax_kernel   max |v| per (b, head, channel) (atomicMax on the
//                               bits of non-negative floats into a zeroed array);
//   skiparse_fwd8_prep_kernel   persistent CTAs (two per SM when their shared
//                               memory fits, one RoPE table copy each) over
//                               (scope, 128-position tile) items: a TMA warp
//                               stages the item's q and k tiles through the scope
//                               gather (one slot per CTA, or a two-slot ring with
//                               one CTA per SM); the compute warps apply RoPE and
//                               quantize q (per row) and k (per tile), quantize v
//                               (read one row group ahead) and transpose it in
//                               shared memory, all in scope-tile order, so the
//                               attention kernel reads plain 128 x 128-byte boxes
//                               (every 8-bit operand K-major);
//   skiparse_fwd8_kernel        two Q tiles per CTA as the bf16 forward (softmax
//   skiparse_fwdm8_kernel       warps 0-7, TMA warp 8), kind::f8f6f4 MMAs (4 per
//                               128 x 128 product instead of 8; the mixed recipe's
//                               S as 8 kind::f16 MMAs) issued by one warp per Q
//                               tile (9, 10); P as E4M3 codes in shared memory, so
//                               S of the next K tile is issued as soon as the
//                               softmax warps hold S in registers.
#include "skiparse_internal.h"

namespace skp {

namespace {

constexpr int kD8 = 128;
constexpr int kF8Threads = 352;   // softmax 0-7, TMA 8, MMA issuers 9 (Q tile A) and 10 (Q tile B)
constexpr int kPrepComputeWarps = 8;
constexpr int kPrepThreads = (kPrepComputeWarps + 1) * 32;   // 8 compute warps, then the TMA warp
constexpr int kPrepCompute = kPrepComputeWarps * 32;
constexpr int kPrepHalf = 128 * 128;                          // 128 rows x 64 bf16 channels, 128-byte swizzle
constexpr int kPrepStage = 4 * kPrepHalf;                     // q and k tiles, two channel halves each
constexpr float kE4M3Max = 448.0f;
constexpr float kInt8Max = 127.0f;

// bytes of one 128-channel row of q / k codes: E4M3 (1 byte each) or INT8
// codes held as bf16 integers (2 bytes each, the operands of a kind::f16 MMA)
__host__ __device__ constexpr int qk_row_bytes(bool si8) { return si8 ? 256 : 128; }

// two INT8 codes RNE(a), RNE(b) (clamped to +-127) as a bf16 pair
__device__ __forceinline__ uint32_t i8x2_bf16(float a, float b) {
  return pack_bf16(fminf(fmaxf(rintf(a), -kInt8Max), kInt8Max), fminf(fmaxf(rintf(b), -kInt8Max), kInt8Max));
}

// The prep kernel's own shared-memory layout of the RoPE table (D = 128).
// Lane class cb = 0..7 of a row rotates the channel pairs 8 cb .. 8 cb + 7,
// which lie on one axis (cb 0-1: t, 2-4: h, 5-7: w) and take 64 bytes of the
// global table per axis position. In that table every such run starts on a
// 64-byte boundary, so the 8 lanes of a row read only two 16-byte bank groups
// at a time (4-way conflicts). Here two classes share each 128-byte line:
// region 0 holds classes 0 and 1 (line = lb[0] + t), region 1 classes 2 and 3
// (lb[1] + h), region 2 classes 5 and 6 (lb[2] + w), region 3 classes 4 (h)
// and 7 (w), line lb[3] + position; a region's lines number its longer axis,
// so only region 3 leaves half-lines unused (|H - W| of them). Class cb of
// region c starts at unit sigma = c (first class) or c + 4 (second), and its
// 16-byte unit m' (pairs 2 m', 2 m' + 1 of its 8) sits at unit
// (sigma + (m' ^ 2 (cb >> 2))) & 7 of the line: at step m a lane reads unit
// (sigma + m) & 7, a different bank group for each of the 8 lanes. (The
// m' ^ 2 (cb >> 2) matches the order in which lanes 4-7 read their staged
// q / k chunks, second chunk first.)
// 4-bit fields, index cb: region, sigma; index c: the region's two classes
constexpr uint32_t kTabRegion = 0x32231100u, kTabSigma = 0x76235140u;
constexpr uint32_t kTabFirst = 0x4520u, kTabSecond = 0x7631u;

__host__ __device__ __forceinline__ int nibble(uint32_t x, int i) { return (int)((x >> (4 * i)) & 15u); }

struct PrepTab { int lb[4]; int lines; };

__host__ __device__ inline PrepTab prep_tab(int T, int H, int W) {
  PrepTab t;
  t.lb[0] = 0;
  t.lb[1] = T;
  t.lb[2] = T + H;
  t.lb[3] = T + H + W;
  t.lines = t.lb[3] + (H > W ? H : W);
  return t;
}

// first line of region c (selects, not an indexed load from a local array)
__host__ __device__ __forceinline__ int prep_lb(const PrepTab& t, int c) {
  return c == 0 ? t.lb[0] : (c == 1 ? t.lb[1] : (c == 2 ? t.lb[2] : t.lb[3]));
}

__host__ __device__ inline size_t prep_table_bytes(int T, int H, int W) { return (size_t)prep_tab(T, H, W).lines * 128; }

// prep kernel shared memory: 1 KB header (barriers, per-warp maxima, abort
// flag), the staging ring (1024-byte aligned for the swizzle), the V^T
// transpose buffer (128 channels x 32 words), the RoPE table
__host__ __device__ inline size_t prep_smem(int stages, int T, int H, int W) {
  return 1024 + (size_t)stages * kPrepStage + (size_t)128 * 32 * 4 + prep_table_bytes(T, H, W);
}

// copies the global table (built once per call) into the layout above
__device__ __forceinline__ void prep_load_table(float4* tab, const float2* gtab, const RopeParams& r, const PrepTab& pt,
                                                int tid, int nthreads) {
  for (int u = tid; u < pt.lines * 8; u += nthreads) {
    const int line = u >> 3, slot = u & 7;
    const int c = line >= pt.lb[3] ? 3 : (line >= pt.lb[2] ? 2 : (line >= pt.lb[1] ? 1 : 0));
    const int j = (slot - c) & 7;                       // 0-3: first class, 4-7: second
    const int cb = nibble(j < 4 ? kTabFirst : kTabSecond, c);
    const int mp = (j & 3) ^ (2 * (cb >> 2));
    const int pos = line - prep_lb(pt, c);
    const PairSel sel = pair_select(r, 8 * cb);
    const int npos = sel.axis == 0 ? r.T : (sel.axis == 1 ? r.H : r.W);
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pos < npos) val = __ldg(reinterpret_cast<const float4*>(gtab + sel.base + pos * sel.stride + sel.local + 2 * mp));
    tab[u] = val;
  }
}

// 2^6 P = 2^(S * ck + off) for one softmax row held in registers (x, 128 keys;
// off = 6 - m), as E4M3 codes: word w of pk holds keys 4w .. 4w+3, the first
// in the lowest byte. Returns the row sum of the unquantized 2^6 P. With
// RAGGED, keys at or past `valid` get P = 0.
template <bool RAGGED>
__device__ __forceinline__ float softmax_p_e4m3(const float (&x)[kTile], uint32_t (&pk)[kTile / 4], float ck,
                                                float off, int valid) {
  const unsigned long long ck2 = f2_pack(ck, ck);
  const unsigned long long off2 = f2_pack(off, off);
  unsigned long long acc2[2] = {0ull, 0ull};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k0 = c * 32 + 4 * e;
      float t0, t1, t2, t3;
      f2_unpack(ffma2(f2_pack(x[k0], x[k0 + 1]), ck2, off2), t0, t1);
      f2_unpack(ffma2(f2_pack(x[k0 + 2], x[k0 + 3]), ck2, off2), t2, t3);
      float p0 = ex2(t0), p1 = ex2(t1), p2 = ex2(t2), p3 = ex2(t3);
      if constexpr (RAGGED) {
        p0 = k0 < valid ? p0 : 0.f;
        p1 = k0 + 1 < valid ? p1 : 0.f;
        p2 = k0 + 2 < valid ? p2 : 0.f;
        p3 = k0 + 3 < valid ? p3 : 0.f;
      }
      acc2[0] = fadd2(acc2[0], f2_pack(p0, p1));
      acc2[1] = fadd2(acc2[1], f2_pack(p2, p3));
      pk[c * 8 + e] = e4m3x4(p0, p1, p2, p3);
    }
  }
  float s0, s1, s2, s3;
  f2_unpack(acc2[0], s0, s1);
  f2_unpack(acc2[1], s2, s3);
  return (s0 + s1) + (s2 + s3);
}

template <bool SI8>
struct F8Layout {
  static constexpr int TILE = 128 * 128;          // 16 KB: 128 rows x 128 bytes, one 128-byte swizzled box
  static constexpr int QK = 128 * qk_row_bytes(SI8);   // a Q or K tile: one E4M3 box, or two bf16 boxes
  static constexpr int HDR = 1024;
  static constexpr int QA_OFF = HDR;
  static constexpr int QB_OFF = QA_OFF + QK;
  static constexpr int K_OFF = QB_OFF + QK;
  static constexpr int V_OFF = K_OFF + 2 * QK;
  static constexpr int PA_OFF = V_OFF + 2 * TILE;   // P of Q tile A as E4M3 codes (A operand of P V)
  static constexpr int PB_OFF = PA_OFF + TILE;
  static constexpr int BYTES = PB_OFF + TILE;
};

enum F8Bar {
  E_QFULL, E_QEMPTY,
  E_KFULL0, E_KFULL1, E_KEMPTY0, E_KEMPTY1,
  E_VFULL0, E_VFULL1, E_VEMPTY0, E_VEMPTY1,
  E_SFULL_A, E_SFULL_B, E_PFULL_A, E_PFULL_B, E_ODONE_A, E_ODONE_B, E_OEMPTY_A, E_OEMPTY_B,
  E_SFREE_A, E_SFREE_B,   // the softmax warps hold S in registers: the next S may be written
  E_FINAL, E_NBARS
};

}  // namespace

// ---------------------------------------------------------------------------
// max |v| per (b, head, channel): grid (B * heads, token chunks of 256), (b, head)
// fastest so that blocks running together read whole token rows of v. A
// half-warp reads one 256-byte (token, head) row per load, 16 bytes a lane, and
// each lane keeps eight rows in flight: short sequences give each block little
// work, so the loads in flight, not the bytes, set the pace.
// ---------------------------------------------------------------------------
constexpr int kVmaxThreads = 256;

__global__ void __launch_bounds__(kVmaxThreads) skiparse_fwd8_vmax_kernel(const __grid_constant__ Fwd8Params p) {
  constexpr int kWarps = kVmaxThreads / 32;
  __shared__ float part[kWarps][kD8];
  const Geom& g = p.g;
  const int bh = blockIdx.x;
  const int b = bh / g.heads, head = bh - b * g.heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = lane >> 4, c8 = lane & 15;          // row of the pair, group of 8 channels
  const int t0 = blockIdx.y * 256;
  const int t1 = min(t0 + 256, g.N);
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = 0.f;
  // rows t0 + 16 j + 2 warp + hw, j = 0..15, in two batches of eight loads
#pragma unroll
  for (int j0 = 0; j0 < 16; j0 += 8) {
    uint4 u[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // rows past the end read the chunk's last row again (a max ignores repeats),
      // so the loads carry no branch and all eight issue back to back
      const int i = min(t0 + 16 * (j0 + j) + 2 * warp + hw, t1 - 1);
      u[j] = __ldg(reinterpret_cast<const uint4*>(p.v + (((size_t)b * g.N + i) * g.heads + head) * kD8 + c8 * 8));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w4[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mx[2 * e] = fmaxf(mx[2 * e], fabsf(bf16lo(w4[e])));
        mx[2 * e + 1] = fmaxf(mx[2 * e + 1], fabsf(bf16hi(w4[e])));
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
  if (hw == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) part[warp][c8 * 8 + e] = mx[e];
  }
  __syncthreads();
  if (threadIdx.x < kD8) {
    const int d = threadIdx.x;
    float m = part[0][d];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, part[w][d]);
    atomicMax(p.vmax + (size_t)bh * kD8 + d, __float_as_uint(m));   // non-negative floats order as their bits
  }
}

// ---------------------------------------------------------------------------
// prep: persistent CTAs (one per SM, one RoPE table each) over (scope index
// sidx = (b * heads + head) * k + s, 128-position tile) items. The TMA warp
// stages each item's q and k tiles (bf16, through the scope gather: smem row r
// is scope position tile * 128 + r) in a ring of prep_stages slots, so the
// next tiles load while the compute warps work on this one (two CTAs per SM
// when their shared memory fits: one slot each); v rows are read directly, a
// group of four rows ahead.
template <bool SI8>
__device__ __forceinline__ void fwd8_prep(const Fwd8Params& p) {
  constexpr float QMAX = SI8 ? kInt8Max : kE4M3Max;
  constexpr int QROW = qk_row_bytes(SI8);
  extern __shared__ __align__(1024) uint8_t psm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(psm) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.err, 0, ERR_SMEM_ALIGN);
    return;
  }
  const Geom& g = p.g;
  const int stages = p.prep_stages;
  float* rowmax = reinterpret_cast<float*>(psm + 64);                               // one per compute warp
  int* abort_flag = reinterpret_cast<int*>(psm + 192);
  uint8_t* ring = psm + 1024;
  uint32_t* vt = reinterpret_cast<uint32_t*>(ring + (size_t)stages * kPrepStage);  // 128 channels x 32 words
  float4* tab = reinterpret_cast<float4*>(vt + kD8 * 32);                           // RoPE table
  const uint32_t bar0 = smem_u32(psm);
  // barriers: FULL of slot st at st, EMPTY of slot st at 2 + st
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  constexpr int E = ERR_KERNEL_FWD + 0xC0;
  const Ctl ctl{abort_flag, p.err};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int st = 0; st < stages; ++st) {
      mbar_init(bar(st), 1);
      mbar_init(bar(2 + st), kPrepComputeWarps);
    }
    mbar_fence_init();
  }
  pdl_trigger();                                     // the attention kernel may take SMs as this pass drains
  pdl_wait();                                        // the cos/sin table (and the v maxima before it) are complete
  const PrepTab pt = prep_tab(p.rope.T, p.rope.H, p.rope.W);
  prep_load_table(tab, p.rope_gtab, p.rope, pt, threadIdx.x, blockDim.x);
  __syncthreads();
  const int n_items = g.B * g.heads * g.ks * g.n_tiles;
  // head fastest: the CTAs working at the same time read all heads of the same
  // tokens, i.e. whole (token, heads x D) rows of q, k and v, not one head's
  // 256-byte slice of every row. Only the call's ks scopes s0, s0 + sstep, ...
  auto decode = [&](int item, int& tile, int& s, int& sidx, int& b, int& head) {
    head = item % g.heads;
    const int rest = item / g.heads;
    tile = rest % g.n_tiles;
    const int bs = rest / g.n_tiles;
    s = g.s0 + (bs % g.ks) * g.sstep;
    b = bs / g.ks;
    sidx = (b * g.heads + head) * g.k + s;
  };

  if (warp == kPrepComputeWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      uint32_t issued[2] = {0, 0};
      int it = 0;
      for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
        const int st = it % stages;
        const int n = it / stages;
        if (n > 0 && !mbar_wait(bar(2 + st), (n - 1) & 1, ctl, E + 2 + st)) break;
        int tile, s, sidx, b, head;
        decode(item, tile, s, sidx, b, head);
        const uint32_t dst = smem_u32(ring + (size_t)st * kPrepStage);
        // through the scope gather, or (unequal scopes) the scope-ordered copies
        const TileCoord tc = scope_tile(g, s, b, tile * kTile);
        mbar_expect_tx(bar(st), kPrepStage);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          load_tile(dst + h * kPrepHalf, &p.tm_q, bar(st), tc, h * 64, head);
          load_tile(dst + (2 + h) * kPrepHalf, &p.tm_k, bar(st), tc, h * 64, head);
        }
        ++issued[st];
      }
      // copies still in flight (only after an abort) must land before exit
      for (int st = 0; st < stages; ++st)
        if (issued[st]) mbar_drain(bar(st), (issued[st] - 1) & 1);
    }
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------ compute warps
  // Warp w owns the tile's rows 4(w + 8 i) + rq, rq = 0..3, i = 0..3.
  // q and k (staged): lane l takes row rq = l / 8 of each group and channels
  // 16 cb .. 16 cb + 15, cb = l % 8 (pairs 8 cb .. 8 cb + 7, all in one RoPE
  // chunk, contiguous in the table), so per-row work (token coordinates, table
  // index, the row max over 8 lanes, the scale divisions) serves four rows per
  // instruction. In a staged row those channels are the 16-byte chunks
  // 2 (cb % 4) and 2 (cb % 4) + 1 of half cb / 4, each XOR (row % 8); lanes
  // 4-7 (hsel = 1) read the second chunk first, so that the two halves' lanes
  // fall on different bank groups. Their registers then hold pairs 4-7 before
  // 0-3, which the table layout and the code stores undo.
  // v (read directly): lane l takes channels 4 l .. 4 l + 3 of all four rows,
  // the layout the V^T transpose needs.
  const int rq = lane >> 3, cb = lane & 7;
  const int hsel = cb >> 2;
  const uint32_t half_off = (uint32_t)hsel * kPrepHalf;
  const uint32_t chunk_a = (uint32_t)(2 * (cb & 3) + hsel), chunk_b = (uint32_t)(2 * (cb & 3) + 1 - hsel);
  // this lane's table lines: region of its class, axis that indexes it
  const int tab_axis = pair_select(p.rope, 8 * cb).axis;   // D = 128: pairs 0-15 t, 16-39 h, 40-63 w
  const float4* tab_lane = tab + (size_t)prep_lb(pt, nibble(kTabRegion, cb)) * 8;
  const int tab_sigma = nibble(kTabSigma, cb);
  auto load_v = [&](int tile, int s, int Ls, int b, int head, int i, uint2 (&vv)[4]) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int pos = tile * kTile + 4 * (warp + 8 * i) + rr;
      vv[rr] = make_uint2(0u, 0u);
      if (pos < Ls) {
        const int tok = token_of(g, s, pos);
        vv[rr] = __ldg(reinterpret_cast<const uint2*>(p.v + (((size_t)b * g.N + tok) * g.heads + head) * kD8 + lane * 4));
      }
    }
  };
  int it = 0;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const int st = it % stages;
    int tile, s, sidx, b, head;
    decode(item, tile, s, sidx, b, head);
    const int bh = sidx / g.k;
    const int Ls = scope_len(g, s);                  // rows at or past it get zero codes
    uint2 vcur[4];
    load_v(tile, s, Ls, b, head, 0, vcur);           // in flight while the staged tiles land
    float inv_v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float m = __uint_as_float(p.vmax[(size_t)bh * kD8 + lane * 4 + e]);
      inv_v[e] = m > 0.f ? kE4M3Max / m : 0.f;
    }
    if (!bar_and<1, kPrepCompute>(mbar_wait(bar(st), (it / stages) & 1, ctl, E + st))) break;
    const uint8_t* q_tile = ring + (size_t)st * kPrepStage;
    const uint8_t* k_tile = q_tile + 2 * kPrepHalf;
    // k in two passes over the staged tile: the tile's max |k| first, the codes
    // once it is known (rotating again instead of holding 64 values per thread)
    float kmax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r0 = 4 * (warp + 8 * i);
      uint2 vnext[4] = {};
      if (i < 3) load_v(tile, s, Ls, b, head, i + 1, vnext);
      // ---- q and k of row r0 + rq, channels 16 cb .. 16 cb + 15
      {
        const int r = r0 + rq;
        const int pos = tile * kTile + r;
        const size_t slot = (size_t)sidx * p.Lp + pos;          // scope-order row
        const bool valid = pos < Ls;                 // not warp-uniform: four rows per warp
        uint4 qc = make_uint4(0u, 0u, 0u, 0u), qc2 = make_uint4(0u, 0u, 0u, 0u);
        float sq = 0.f;
        float qr[16];
        float qm = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) qr[e] = 0.f;
        if (valid) {
          const uint32_t rb = (uint32_t)r * 128u + half_off;
          const uint32_t o0 = rb + ((chunk_a ^ (uint32_t)(r & 7)) << 4);
          const uint32_t o1 = rb + ((chunk_b ^ (uint32_t)(r & 7)) << 4);
          uint32_t qw[8], kw[8];
          *reinterpret_cast<uint4*>(qw) = *reinterpret_cast<const uint4*>(q_tile + o0);
          *reinterpret_cast<uint4*>(qw + 4) = *reinterpret_cast<const uint4*>(q_tile + o1);
          *reinterpret_cast<uint4*>(kw) = *reinterpret_cast<const uint4*>(k_tile + o0);
          *reinterpret_cast<uint4*>(kw + 4) = *reinterpret_cast<const uint4*>(k_tile + o1);
          int t, hh, w;
          token_coords(p.rope, token_of(g, s, pos), t, hh, w);
          const int apos = tab_axis == 0 ? t : (tab_axis == 1 ? hh : w);
          const float4* tp = tab_lane + apos * 8;
#pragma unroll
          for (int m2 = 0; m2 < 4; ++m2) {
            const float4 cs = tp[(tab_sigma + m2) & 7];            // the pairs of words 2 m2, 2 m2 + 1
            const float2 qa = rope_rotate(bf16lo(qw[2 * m2]), bf16hi(qw[2 * m2]), make_float2(cs.x, cs.y));
            const float2 qb = rope_rotate(bf16lo(qw[2 * m2 + 1]), bf16hi(qw[2 * m2 + 1]), make_float2(cs.z, cs.w));
            const float2 ka = rope_rotate(bf16lo(kw[2 * m2]), bf16hi(kw[2 * m2]), make_float2(cs.x, cs.y));
            const float2 kb = rope_rotate(bf16lo(kw[2 * m2 + 1]), bf16hi(kw[2 * m2 + 1]), make_float2(cs.z, cs.w));
            qr[4 * m2 + 0] = qa.x; qr[4 * m2 + 1] = qa.y; qr[4 * m2 + 2] = qb.x; qr[4 * m2 + 3] = qb.y;
            qm = fmaxf(qm, fmaxf(fmaxf(fabsf(qa.x), fabsf(qa.y)), fmaxf(fabsf(qb.x), fabsf(qb.y))));
            kmax = fmaxf(kmax, fmaxf(fmaxf(fabsf(ka.x), fabsf(ka.y)), fmaxf(fabsf(kb.x), fabsf(kb.y))));
          }
        }
        // q: per-row scale, the row's max over its 8 lanes (every lane takes part)
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
        if (valid) {
          const float qi = qm > 0.f ? QMAX / qm : 0.f;
          if constexpr (SI8) {
            qc.x = i8x2_bf16(qr[0] * qi, qr[1] * qi);
            qc.y = i8x2_bf16(qr[2] * qi, qr[3] * qi);
            qc.z = i8x2_bf16(qr[4] * qi, qr[5] * qi);
            qc.w = i8x2_bf16(qr[6] * qi, qr[7] * qi);
            qc2.x = i8x2_bf16(qr[8] * qi, qr[9] * qi);
            qc2.y = i8x2_bf16(qr[10] * qi, qr[11] * qi);
            qc2.z = i8x2_bf16(qr[12] * qi, qr[13] * qi);
            qc2.w = i8x2_bf16(qr[14] * qi, qr[15] * qi);
          } else {
            qc.x = e4m3x4(qr[0] * qi, qr[1] * qi, qr[2] * qi, qr[3] * qi);
            qc.y = e4m3x4(qr[4] * qi, qr[5] * qi, qr[6] * qi, qr[7] * qi);
            qc.z = e4m3x4(qr[8] * qi, qr[9] * qi, qr[10] * qi, qr[11] * qi);
            qc.w = e4m3x4(qr[12] * qi, qr[13] * qi, qr[14] * qi, qr[15] * qi);
          }
          sq = qm > 0.f ? qm / QMAX : 1.f;
        }
        if constexpr (SI8) {
          // the lane's 32 bytes of the row in one store (the workspace rows are 32-byte aligned)
          const uint4 lo = hsel ? qc2 : qc, hi = hsel ? qc : qc2;
          st_global_32b(p.q8 + slot * QROW + cb * 32, lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w);
        } else {
          *reinterpret_cast<uint4*>(p.q8 + slot * QROW + cb * 16) =
              hsel ? make_uint4(qc.z, qc.w, qc.x, qc.y) : qc;
        }
        if (cb == 0) p.sq[slot] = sq;
      }
      // ---- v of rows r0 .. r0 + 3, channels 4 lane .. 4 lane + 3
      uint32_t vc[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint2 vu = vcur[rr];
        vc[rr] = e4m3x4(bf16lo(vu.x) * inv_v[0], bf16hi(vu.x) * inv_v[1], bf16lo(vu.y) * inv_v[2],
                        bf16hi(vu.y) * inv_v[3]);
      }
      // 4 rows x 4 channels of v codes -> channel 4 lane + e gets positions r0 .. r0+3 in one
      // word, stored at word (r0 / 4) ^ lane of the channel's 32 (conflict-free across lanes)
      const uint32_t lo01 = __byte_perm(vc[0], vc[1], 0x5140), hi01 = __byte_perm(vc[0], vc[1], 0x7362);
      const uint32_t lo23 = __byte_perm(vc[2], vc[3], 0x5140), hi23 = __byte_perm(vc[2], vc[3], 0x7362);
      const int wi = (r0 >> 2) ^ lane;
      vt[(4 * lane + 0) * 32 + wi] = __byte_perm(lo01, lo23, 0x5410);
      vt[(4 * lane + 1) * 32 + wi] = __byte_perm(lo01, lo23, 0x7632);
      vt[(4 * lane + 2) * 32 + wi] = __byte_perm(hi01, hi23, 0x5410);
      vt[(4 * lane + 3) * 32 + wi] = __byte_perm(hi01, hi23, 0x7632);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) vcur[rr] = vnext[rr];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kmax = fmaxf(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    if (lane == 0) rowmax[warp] = kmax;
    asm volatile("bar.sync 2, %0;" :: "n"(kPrepCompute) : "memory");
    float tmax = 0.f;
#pragma unroll
    for (int w = 0; w < kPrepComputeWarps; ++w) tmax = fmaxf(tmax, rowmax[w]);
    const float ki = tmax > 0.f ? QMAX / tmax : 0.f;
    if (threadIdx.x == 0) p.sk[(size_t)sidx * g.n_tiles + tile] = tmax > 0.f ? tmax / QMAX : 1.f;
    // k: one scale per tile; rows past the scope's end get zero codes
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * (warp + 8 * i) + rq;
      const int pos = tile * kTile + r;
      const size_t slot = (size_t)sidx * p.Lp + pos;
      uint4 kc = make_uint4(0u, 0u, 0u, 0u), kc2 = make_uint4(0u, 0u, 0u, 0u);
      if (pos < Ls) {
        const uint32_t rb = (uint32_t)r * 128u + half_off;
        uint32_t kw[8];
        *reinterpret_cast<uint4*>(kw) = *reinterpret_cast<const uint4*>(k_tile + rb + ((chunk_a ^ (uint32_t)(r & 7)) << 4));
        *reinterpret_cast<uint4*>(kw + 4) = *reinterpret_cast<const uint4*>(k_tile + rb + ((chunk_b ^ (uint32_t)(r & 7)) << 4));
        int t, hh, w;
        token_coords(p.rope, token_of(g, s, pos), t, hh, w);
        const int apos = tab_axis == 0 ? t : (tab_axis == 1 ? hh : w);
        const float4* tp = tab_lane + apos * 8;
        uint32_t* kcw = reinterpret_cast<uint32_t*>(&kc);
        uint32_t* kcw2 = reinterpret_cast<uint32_t*>(&kc2);
#pragma unroll
        for (int m2 = 0; m2 < 4; ++m2) {
          const float4 cs = tp[(tab_sigma + m2) & 7];
          const float2 ka = rope_rotate(bf16lo(kw[2 * m2]), bf16hi(kw[2 * m2]), make_float2(cs.x, cs.y));
          const float2 kb = rope_rotate(bf16lo(kw[2 * m2 + 1]), bf16hi(kw[2 * m2 + 1]), make_float2(cs.z, cs.w));
          if constexpr (SI8) {
            // register channels 4 m2 .. 4 m2 + 3 of this lane's 16: words 2 m2, 2 m2 + 1 of 8
            uint32_t* w = m2 < 2 ? kcw : kcw2;
            w[(2 * m2) & 3] = i8x2_bf16(ka.x * ki, ka.y * ki);
            w[(2 * m2 + 1) & 3] = i8x2_bf16(kb.x * ki, kb.y * ki);
          } else {
            kcw[m2] = e4m3x4(ka.x * ki, ka.y * ki, kb.x * ki, kb.y * ki);
          }
        }
      }
      if constexpr (SI8) {
        const uint4 lo = hsel ? kc2 : kc, hi = hsel ? kc : kc2;
        st_global_32b(p.k8 + slot * QROW + cb * 32, lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w);
      } else {
        *reinterpret_cast<uint4*>(p.k8 + slot * QROW + cb * 16) = hsel ? make_uint4(kc.z, kc.w, kc.x, kc.y) : kc;
      }
    }
    // this warp has read its rows of the staged q / k for the last time: the
    // slot may be refilled
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(2 + st));
    // V^T rows: channel d of this tile's 128 positions, one word per thread per step
    for (int idx = threadIdx.x; idx < kD8 * 32; idx += kPrepCompute) {
      const int d = idx >> 5, c = idx & 31;
      const uint32_t word = vt[d * 32 + (c ^ (d >> 2))];
      *reinterpret_cast<uint32_t*>(p.vt8 + ((size_t)sidx * kD8 + d) * p.Lp + tile * kTile + c * 4) = word;
    }
    asm volatile("bar.sync 3, %0;" :: "n"(kPrepCompute) : "memory");   // vt and rowmax are reused next
  }
}

__global__ void __launch_bounds__(kPrepThreads, 2) skiparse_fwd8_prep_kernel(const __grid_constant__ Fwd8Params p) {
  fwd8_prep<false>(p);
}
__global__ void __launch_bounds__(kPrepThreads, 2) skiparse_fwdm8_prep_kernel(const __grid_constant__ Fwd8Params p) {
  fwd8_prep<true>(p);
}

// ---------------------------------------------------------------------------
// attention over 8-bit operands
// ---------------------------------------------------------------------------
template <bool SI8>
__device__ __forceinline__ void fwd8_attention(const Fwd8Params& p) {
  using Ly = F8Layout<SI8>;
  constexpr int D = kD8;
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
  const uint32_t sPA = smem_u32(smem + Ly::PA_OFF);
  const uint32_t sPB = smem_u32(smem + Ly::PB_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
  const Ctl ctl{abort_flag, p.err};
  const Geom& g = p.g;
  const int n_pairs = (g.n_tiles + 1) >> 1;
  constexpr int E = ERR_KERNEL_FWD + 0x80;
  // unit u = (scope index sidx, Q-tile pair); false for a pair past a shorter
  // scope's end (every role skips it alike)
  auto unit_of = [&](int u, int& pair, int& sidx, int& nt, int& Ls) -> bool {
    pair = u % n_pairs;
    const int r = u / n_pairs;                       // (b, head) * ks + the call's scope number
    const int s = g.s0 + (r % g.ks) * g.sstep;
    sidx = (r / g.ks) * g.k + s;
    nt = scope_tiles(g, s);
    Ls = scope_len(g, s);
    return 2 * pair < nt;
  };

  if (tid == 0) {
    *abort_flag = 0;
    // stages shared by both Q tiles are released by a commit from each MMA issuer
    const uint32_t counts[E_NBARS] = {1, 2, 1, 1, 2, 2, 1, 1, 2, 2, 1, 1, 4, 4, 1, 1, 4, 4, 4, 4, 2};
    for (int i = 0; i < E_NBARS; ++i) mbar_init(bar(i), counts[i]);
    mbar_fence_init();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();                                        // the prep kernel's codes and scales are complete
  auto warp_wait = [&](int i, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar(i), parity, ctl, E + i)) != 0;
  };
  const bool leader = lane == 0;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (leader) {
      tma_prefetch_map(&p.tm_q8);
      tma_prefetch_map(&p.tm_k8);
      tma_prefetch_map(&p.tm_vt);
    }
    uint32_t q_issued = 0, k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
    uint32_t gk = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int pair, sidx, nt, Ls;
      if (!unit_of(u, pair, sidx, nt, Ls)) continue;
      if (it > 0 && !warp_wait(E_QEMPTY, (it - 1) & 1)) break;
      if (leader) {
        mbar_expect_tx(bar(E_QFULL), 2 * Ly::QK);
        if constexpr (SI8) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_load_3d(sQA + h * kHalfBytes, &p.tm_q8, bar(E_QFULL), h * 64, 2 * pair * kTile, sidx);
            tma_load_3d(sQB + h * kHalfBytes, &p.tm_q8, bar(E_QFULL), h * 64, (2 * pair + 1) * kTile, sidx);
          }
        } else {
          tma_load_3d(sQA, &p.tm_q8, bar(E_QFULL), 0, 2 * pair * kTile, sidx);
          tma_load_3d(sQB, &p.tm_q8, bar(E_QFULL), 0, (2 * pair + 1) * kTile, sidx);
        }
      }
      __syncwarp();
      ++q_issued;
      // the next unit's Q codes, prefetched into L2 a few K tiles before this
      // unit ends so that its Q load hits L2
      int npair = 0, nsidx = 0, nnt = 0, nLs = 0;
      bool next = false;
      for (int u2 = u + gridDim.x; u2 < p.n_units; u2 += gridDim.x)
        if (unit_of(u2, npair, nsidx, nnt, nLs)) {
          next = true;
          break;
        }
      const int pf_at = nt > 4 ? nt - 4 : 0;
      for (int j = 0; j < nt; ++j) {
        const uint32_t gg = gk + j;
        const int st = gg & 1;
        const uint32_t n = gg >> 1;
        if (leader && next && j == pf_at) {
#pragma unroll
          for (int h = 0; h < (SI8 ? 2 : 1); ++h)
#pragma unroll
            for (int x = 0; x < 2; ++x)
              asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                           :: "l"((uint64_t)&p.tm_q8), "r"(h * 64), "r"((2 * npair + x) * kTile), "r"(nsidx)
                           : "memory");
        }
        if (n > 0 && !warp_wait(E_KEMPTY0 + st, (n - 1) & 1)) { ok = false; break; }
        if (leader) {
          mbar_expect_tx(bar(E_KFULL0 + st), Ly::QK);
          if constexpr (SI8) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sK + st * Ly::QK + h * kHalfBytes, &p.tm_k8, bar(E_KFULL0 + st), h * 64, j * kTile, sidx);
          } else {
            tma_load_3d(sK + st * Ly::QK, &p.tm_k8, bar(E_KFULL0 + st), 0, j * kTile, sidx);
          }
        }
        __syncwarp();
        ++k_issued[st];
        if (n > 0 && !warp_wait(E_VEMPTY0 + st, (n - 1) & 1)) { ok = false; break; }
        if (leader) {
          mbar_expect_tx(bar(E_VFULL0 + st), Ly::TILE);
          tma_load_3d(sV + st * Ly::TILE, &p.tm_vt, bar(E_VFULL0 + st), j * kTile, 0, sidx);
        }
        __syncwarp();
        ++v_issued[st];
      }
      gk += nt;
      ++it;
    }
    if (leader) {
      if (q_issued) mbar_drain(bar(E_QFULL), (q_issued - 1) & 1);
      for (int st = 0; st < 2; ++st) {
        if (k_issued[st]) mbar_drain(bar(E_KFULL0 + st), (k_issued[st] - 1) & 1);
        if (v_issued[st]) mbar_drain(bar(E_VFULL0 + st), (v_issued[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // One warp per Q tile X (9: A, 10: B), each issuing its own S_X and P_X V
    // (two issuing threads keep the tensor core fed; one alone spends more
    // cycles per MMA issuing than the MMA runs).
    const int xb = warp - 9;
    constexpr uint32_t kId = idesc_e4m3(128, 128);
    constexpr uint32_t kIdS = SI8 ? idesc_bf16(128, 128, false, false) : kId;
    const uint64_t dQ = desc_kmajor(xb ? sQB : sQA, 0);
    const uint64_t dK0 = desc_kmajor(sK, 0), dK1 = desc_kmajor(sK + Ly::QK, 0);
    const uint64_t dV0 = desc_kmajor(sV, 0), dV1 = desc_kmajor(sV + Ly::TILE, 0);
    const uint64_t dP = desc_kmajor(xb ? sPB : sPA, 0);
    const uint32_t colS = xb ? 128u : 0u;
    const uint32_t colO = 256u + (xb ? (uint32_t)D : 0u);
    const int barSF = xb ? E_SFREE_B : E_SFREE_A;
    const int barS = xb ? E_SFULL_B : E_SFULL_A;
    const int barP = xb ? E_PFULL_B : E_PFULL_A;
    const int barO = xb ? E_ODONE_B : E_ODONE_A;
    const int barOE = xb ? E_OEMPTY_B : E_OEMPTY_A;
    // S_X = Q_X K_g^T: 4 E4M3 k-steps of 32 channels, or 8 bf16 k-steps of 16
    // channels over INT8-valued codes (exact integer sums in fp32)
    auto issue_s = [&](int st) {
      const uint64_t dk = st ? dK1 : dK0;
      if constexpr (SI8) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss(tmem + colS, kmajor_step(dQ, ks), kmajor_step(dk, ks), kIdS, ks > 0 ? 1u : 0u);
      } else {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma8_ss(tmem + colS, kmajor_step(dQ, ks), kmajor_step(dk, ks), kIdS, ks > 0 ? 1u : 0u);
      }
    };
    // O_X += P_X V_g: P_X as E4M3 codes in shared memory (K-major), V^T K-major
    auto issue_pv = [&](int st, bool first) {
      const uint64_t dv = st ? dV1 : dV0;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma8_ss(tmem + colO, kmajor_step(dP, ks), kmajor_step(dv, ks), kId, (!first || ks > 0) ? 1u : 0u);
    };
    // Per K step g of a unit: S_X(g+1) as soon as the softmax warps hold S_X(g)
    // in registers, then P_X(g) V once P is in shared memory; the next S is
    // computed while the softmax works on this one.
    uint32_t g0 = 0;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int pair, sidx, n, Ls;
      if (!unit_of(u, pair, sidx, n, Ls)) continue;
      if (!warp_wait(E_QFULL, it & 1)) break;
      if (!warp_wait(E_KFULL0 + (g0 & 1), (g0 >> 1) & 1)) break;
      if (g0 > 0 && !warp_wait(barSF, (g0 - 1) & 1)) break;
      tc_fence_after();
      if (leader) {
        issue_s(g0 & 1);
        tc_commit(bar(barS));
        tc_commit(bar(E_KEMPTY0 + (g0 & 1)));
        if (n == 1) tc_commit(bar(E_QEMPTY));
      }
      __syncwarp();
      for (int j = 0; j < n; ++j) {
        const uint32_t gg = g0 + j;
        const int st = gg & 1;
        const uint32_t nn = gg >> 1;
        if (j + 1 < n) {
          const int st1 = (gg + 1) & 1;
          if (!warp_wait(barSF, gg & 1)) { ok = false; break; }
          if (!warp_wait(E_KFULL0 + st1, ((gg + 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          if (leader) {
            issue_s(st1);
            tc_commit(bar(barS));
            tc_commit(bar(E_KEMPTY0 + st1));
            if (j + 2 == n) tc_commit(bar(E_QEMPTY));
          }
          __syncwarp();
        }
        if (j == 0 && it > 0 && !warp_wait(barOE, (it - 1) & 1)) { ok = false; break; }
        if (!warp_wait(barP, gg & 1)) { ok = false; break; }
        if (!warp_wait(E_VFULL0 + st, nn & 1)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          issue_pv(st, j == 0);
          tc_commit(bar(barO));
          tc_commit(bar(E_VEMPTY0 + st));
        }
        __syncwarp();
      }
      g0 += n;
      ++it;
    }
    if (leader) {
      tc_commit(bar(E_FINAL));
      mbar_drain(bar(E_FINAL), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps (A: 0-3, B: 4-7)
    const int wg = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = wg ? 128u : 0u;
    const uint32_t colO = 256u + (wg ? (uint32_t)D : 0u);
    const int barS = wg ? E_SFULL_B : E_SFULL_A;
    const int barP = wg ? E_PFULL_B : E_PFULL_A;
    const int barO = wg ? E_ODONE_B : E_ODONE_A;
    const int barOE = wg ? E_OEMPTY_B : E_OEMPTY_A;
    const int barSF = wg ? E_SFREE_B : E_SFREE_A;
    // this thread's row of P (128 codes, 128-byte swizzled rows as TMA writes them)
    uint8_t* prow_smem = smem + (wg ? Ly::PB_OFF : Ly::PA_OFF) + r * 128;
    uint32_t g0 = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      int pair, sidx, nt, Ls;
      if (!unit_of(u, pair, sidx, nt, Ls)) continue;
      const int tile = 2 * pair + wg;
      const int prow = tile * kTile + r;
      // scaled score in log2 units = S * sq_row * sk_tile * scale * log2 e
      // (tile B of a scope with an odd tile count lies past Lp: zero rows, no scale)
      const float crow = prow < p.Lp ? p.sq[(size_t)sidx * p.Lp + prow] * p.scale_log2 : 0.f;
      const float* skt = p.sk + (size_t)sidx * g.n_tiles;
      float m = 0.f, l = 0.f;          // l in units of 2^6 P
      for (int j = 0; j < nt; ++j) {
        const uint32_t gg = g0 + j;
        const float ck = crow * __ldg(skt + j);
        if (!mbar_wait(bar(barS), gg & 1, ctl, E + barS)) { ok = false; break; }
        tc_fence_after();
        const int valid = min(kTile, Ls - j * kTile);
        // the whole S row in registers with one TMEM round trip
        float x[kTile];
        tmem_ld128(tmem + lane_base + colS, x);
        // S is in registers: the MMA warp may write the next S over it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(barSF));
        const float mx = (valid == kTile ? row_max128<false>(x, valid) : row_max128<true>(x, valid)) * ck;
        float f = 1.f;
        bool rescale = false;
        // integer reference m, raised to ceil(max) only when the tile's max
        // exceeds it by more than 2: 2^(t - m) < 4, and rescales are powers of two
        if (j == 0) {
          m = ceilf(mx);
        } else {
          const bool need = mx > m + 2.0f;
          rescale = __any_sync(0xffffffffu, need);
          if (rescale) {
            const float m_new = need ? ceilf(mx) : m;
            f = ex2(m - m_new);
            m = m_new;
            l *= f;
          }
        }
        // 2^6 P as E4M3 codes in registers (the full-tile path has no masking)
        uint32_t pk[kTile / 4];
        l += valid == kTile ? softmax_p_e4m3<false>(x, pk, ck, 6.0f - m, valid)
                            : softmax_p_e4m3<true>(x, pk, ck, 6.0f - m, valid);
        // P_X(g-1) V has read the P buffer and added into O: the first PV of a
        // unit follows the previous unit's epilogue, which waited for it
        if (j > 0) {
          if (!mbar_wait(bar(barO), (gg - 1) & 1, ctl, E + barO)) { ok = false; break; }
          tc_fence_after();
        }
        if (rescale) {
          // O *= 2^(m_old - m_new) before P V adds this tile
#pragma unroll 1
          for (int c = 0; c < kD8 / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + lane_base + colO + c * 32, o);
            float oc[16], od[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              oc[e] = o[e] * f;
              od[e] = o[16 + e] * f;
            }
            tmem_st16f(tmem + lane_base + colO + c * 32, oc);
            tmem_st16f(tmem + lane_base + colO + c * 32 + 16, od);
          }
          tmem_st_wait();
        }
        // codes of keys 16c .. 16c+15 are the row's 16-byte chunk c, stored at
        // chunk c ^ (row mod 8) (128-byte swizzle)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow_smem + ((c ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(barP));
      }
      if (!ok) break;
      // ---- epilogue: out = O * s_v / l (l and O both in units of 2^6 P); LSE natural log
      const uint32_t glast = g0 + nt - 1;
      if (!mbar_wait(bar(barO), glast & 1, ctl, E + barO)) break;
      tc_fence_after();
      const int s = sidx % g.k, bh = sidx / g.k;
      const int b = bh / g.heads, head = bh - b * g.heads;
      const bool row_ok = prow < Ls;
      const int tok = row_ok ? token_of(g, s, prow) : 0;
      const float inv_l = 1.0f / (l * kE4M3Max);
      const unsigned* vm = p.vmax + (size_t)bh * D;
      uint16_t* orow = p.out + (((size_t)b * g.N + tok) * g.heads + head) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + lane_base + colO + c * 32, o);
        if (row_ok) {
          // the chunk's 32 per-channel v scales (the same for every row: broadcast loads), 16 bytes at a time
          float sv[32];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(vm + c * 32) + q4);
            sv[4 * q4] = __uint_as_float(u.x);
            sv[4 * q4 + 1] = __uint_as_float(u.y);
            sv[4 * q4 + 2] = __uint_as_float(u.z);
            sv[4 * q4 + 3] = __uint_as_float(u.w);
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16(o[2 * e] * (sv[2 * e] * inv_l), o[2 * e + 1] * (sv[2 * e + 1] * inv_l));
          // rows are D * 2 bytes apart: 32-byte stores whenever out's base allows
          st_global_64b(orow + c * 32, w, (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0);
        }
      }
      if (row_ok) p.lse[((size_t)b * g.heads + head) * g.N + tok] = (m + log2f(l) - 6.0f) * 0.6931471805599453f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(barOE));
      g0 += nt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void __launch_bounds__(kF8Threads, 1) skiparse_fwd8_kernel(const __grid_constant__ Fwd8Params p) {
  fwd8_attention<false>(p);
}
__global__ void __launch_bounds__(kF8Threads, 1) skiparse_fwdm8_kernel(const __grid_constant__ Fwd8Params p) {
  fwd8_attention<true>(p);
}

size_t fwd8_smem_bytes(bool si8) { return si8 ? F8Layout<true>::BYTES : F8Layout<false>::BYTES; }

size_t fwd8_qk_row_bytes(bool si8) { return (size_t)qk_row_bytes(si8); }

int fwd8_prep_stages(int T, int H, int W, size_t optin, size_t smem_sm) {
  const size_t one = prep_smem(1, T, H, W);
  if (one <= optin && 2 * (one + 1024) <= smem_sm) return 1;      // two CTAs per SM overlap their items
  for (int st = 2; st >= 1; --st)
    if (prep_smem(st, T, H, W) <= optin) return st;
  return 0;
}

int fwd8_units(const Geom& g) { return g.B * g.heads * g.ks * ((g.n_tiles + 1) / 2); }

cudaError_t launch_fwd8_vmax(const Fwd8Params& p, cudaStream_t stream) {
  const dim3 grid(p.g.B * p.g.heads, (p.g.N + 255) / 256);
  skiparse_fwd8_vmax_kernel<<<grid, kVmaxThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd8_prep(const Fwd8Params& p, bool si8, int sms, cudaStream_t stream) {
  const size_t smem = prep_smem(p.prep_stages, p.rope.T, p.rope.H, p.rope.W);
  auto kernel = si8 ? skiparse_fwdm8_prep_kernel : skiparse_fwd8_prep_kernel;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = one_wave(kernel, p.g.B * p.g.heads * p.g.ks * p.g.n_tiles, kPrepThreads, smem, sms);
  return launch_after_previous(kernel, grid, kPrepThreads, smem, stream, p);
}

cudaError_t launch_fwd8(const Fwd8Params& p, bool si8, int grid, cudaStream_t stream) {
  const size_t smem = fwd8_smem_bytes(si8);
  auto kernel = si8 ? skiparse_fwdm8_kernel : skiparse_fwd8_kernel;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_after_previous(kernel, grid, kF8Threads, smem, stream, p);
}

}  // namespace skp
