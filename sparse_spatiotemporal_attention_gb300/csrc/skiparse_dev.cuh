// Device building blocks for the Skiparse attention kernels (sm_103a).
//
//  * scope geometry: the token <-> (scope, position) maps of the "Open-Sora
//    Plan" docs page, section "Skiparse Attention" (single and group skip
//    rearrange patterns), written with a group size G: G = 1 for single skip,
//    G = k for group skip. A scope position p holds token
//        i = (p div G) * k * G + s * G + (p mod G),
//    which is i = p*k + s for single skip and i = (p div k)*k^2 + s*k + p mod k
//    for group skip.
//  * 3D RoPE cos/sin table and pair rotation;
//  * thin inline-PTX wrappers: mbarrier, TMA (cp.async.bulk), tcgen05
//    (alloc, mma, commit, ld, st, fences) and the shared-memory / instruction
//    descriptors of tcgen05.mma kind::f16.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace skp {

constexpr int kTile = 128;                  // rows of every Q / K / V tile
constexpr int kHalfBytes = 128 * 128;       // one 128-row x 64-channel bf16 box (128B swizzle)
constexpr int kMaxRopeEntries = 8192;       // cos/sin pairs of the RoPE table
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s per bounded wait

// ---------------------------------------------------------------------------
// Division by a runtime constant d >= 1 for 0 <= n < 2^31, by multiply-high:
// n / d = (n * m) >> (32 + s) with s = ceil(log2 d) and m = floor(2^(32+s) / d) + 1
// (m <= 2^33, so for n < 2^31 the product n * m fits in 64 bits).
// ---------------------------------------------------------------------------
struct FastDiv {
  unsigned long long m;
  int s;
  int d;
};

inline FastDiv make_fastdiv(int d) {
  FastDiv f;
  f.d = d;
  int s = 0;
  while ((1ll << s) < d) ++s;
  f.s = s;
  f.m = (unsigned long long)((((unsigned __int128)1) << (32 + s)) / (unsigned)d) + 1ull;
  return f;
}

__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
  return (int)(((unsigned long long)(unsigned)n * f.m) >> (32 + f.s));
}

// ---------------------------------------------------------------------------
// Geometry and RoPE parameters (plain structs, passed inside kernel params)
// ---------------------------------------------------------------------------

struct Geom {
  int B, heads, N, D;
  int k;        // sparse_k: number of scopes
  int G;        // group size: 1 (single skip) or k (group skip); always a power of two
  int lgG;      // log2(G)
  int L;        // length of the longest scope (scope 0): N / k when k (k^2) divides N
  int Nn;       // L / G: rows of the merged (n, b) tensor-map dimension per batch
  int n_tiles;  // ceil(L / 128): tiles of the longest scope
  int packed;   // 1: q, k, v (dO) are read from scope-ordered copies (k, B, Lp, heads, D)
  int Lp;       // n_tiles * 128: rows per (scope, batch) of the scope-ordered copies
  int Qb, Rb;   // N = Qb * k * G + Rb: whole blocks of k groups, and the tokens left over
  FastDiv fLp;  // division by Lp (scope-ordered row -> (scope, batch), position)
  FastDiv fB;   // division by B
  int s0, sstep, ks;   // the scopes computed: s0, s0 + sstep, ... below k, ks of them (all k by default)
  FastDiv fk;   // division by k
  FastDiv fkG;  // division by k * G
  FastDiv fheads;  // division by heads (row index -> (b * N + token, head))
  FastDiv fN;      // division by N (b * N + token -> (b, token))
};

// (b, token i, head) of row index `row` = (b * N + i) * heads + head of a
// (B, N, heads, D) tensor; rows < 2^31.
__device__ __forceinline__ void row_coords(const Geom& g, int row, int& b, int& i, int& head) {
  const int bi = fdiv(row, g.fheads);
  head = row - bi * g.heads;
  b = fdiv(bi, g.fN);
  i = bi - b * g.N;
}

struct RopeParams {
  double om_t[16];    // rope_theta^(-2j/dt) for the t chunk (dt = D/4 channels, D/8 pairs)
  double om_hw[24];   // rope_theta^(-2j/dh) for the h and w chunks (3D/8 channels each)
  int T, H, W;
  int dt2, dh2;       // pairs per chunk: D/8 and 3D/16
  int entries;        // T*dt2 + H*dh2 + W*dh2
  FastDiv fHW;        // division by H*W
  FastDiv fW;         // division by W
};

// Length of scope s: the tokens i with (i div G) mod k = s. Every block of k
// groups gives each scope G tokens; the Rb tokens of the last, partial block
// fill scope 0's group first, then scope 1's, ... (the last group may be partial).
__host__ __device__ __forceinline__ int scope_len(const Geom& g, int s) {
  const int extra = g.Rb - s * g.G;
  return g.Qb * g.G + (extra < 0 ? 0 : (extra > g.G ? g.G : extra));
}
__host__ __device__ __forceinline__ int scope_tiles(const Geom& g, int s) { return (scope_len(g, s) + 127) >> 7; }

// Whether scope s is among the scopes this call computes (s0 + j * sstep).
__device__ __forceinline__ bool in_subset(const Geom& g, int s) {
  return s >= g.s0 && (g.sstep == 1 || (s - g.s0) % g.sstep == 0);
}

__device__ __forceinline__ int token_of(const Geom& g, int s, int p) {
  return ((p >> g.lgG) * g.k << g.lgG) + (s << g.lgG) + (p & (g.G - 1));
}

__device__ __forceinline__ void scope_pos_of(const Geom& g, int i, int& s, int& p) {
  const int ig = i >> g.lgG;                     // i / G
  s = ig - fdiv(ig, g.fk) * g.k;                 // (i / G) mod k
  p = (fdiv(i, g.fkG) << g.lgG) + (i & (g.G - 1));
}

__device__ __forceinline__ void token_coords(const RopeParams& r, int i, int& t, int& h, int& w) {
  t = fdiv(i, r.fHW);
  const int rem = i - t * r.fHW.d;
  h = fdiv(rem, r.fW);
  w = rem - h * r.W;
}

// Table entry e holds (cos, sin) of pos * omega for one axis, position and pair.
// Angles are reduced modulo 2*pi in double before the float sincos, so large
// positions lose no accuracy.
__device__ __forceinline__ float2 rope_cos_sin(int pos, double om) {
  const double a = (double)pos * om;
  const double n = rint(a * 0.15915494309189535);          // a / (2 pi)
  double red = fma(-n, 6.283185307179586, a);               // 2 pi, high part
  red = fma(-n, 2.4492935982947064e-16, red);               // 2 pi, low part
  float sn, cs;
  sincosf((float)red, &sn, &cs);
  return make_float2(cs, sn);
}

// Entry e of the table: (cos, sin) of position pos times omega_j for one axis.
__host__ __device__ __forceinline__ void rope_entry_args(const RopeParams& r, int e, int& pos, double& om) {
  const int nt = r.T * r.dt2, nh = r.H * r.dh2;
  int j;
  if (e < nt) {
    pos = e / r.dt2; j = e - pos * r.dt2; om = r.om_t[j];
  } else if (e < nt + nh) {
    const int e2 = e - nt; pos = e2 / r.dh2; j = e2 - pos * r.dh2; om = r.om_hw[j];
  } else {
    const int e2 = e - nt - nh; pos = e2 / r.dh2; j = e2 - pos * r.dh2; om = r.om_hw[j];
  }
}

__device__ __forceinline__ void rope_build_table(float2* tab, const RopeParams& r, int tid, int nthreads) {
  for (int e = tid; e < r.entries; e += nthreads) {
    int pos;
    double om;
    rope_entry_args(r, e, pos, om);
    tab[e] = rope_cos_sin(pos, om);
  }
}

// Shared-memory copy of a table built once per call in global memory
// (skiparse_rope_table_kernel), instead of each CTA rebuilding it: the angle
// reduction runs on the FP64 pipe, which a wave of CTAs would otherwise share.
__device__ __forceinline__ void rope_load_table(float2* tab, const float2* gtab, int entries, int tid, int nthreads) {
  for (int e = tid; e < entries; e += nthreads) tab[e] = __ldg(gtab + e);
}

// Which table slice a channel pair pp (0 .. D/2-1) reads from.
struct PairSel { int base, stride, local, axis; };

__device__ __forceinline__ PairSel pair_select(const RopeParams& r, int pp) {
  PairSel s;
  if (pp < r.dt2) { s.base = 0; s.stride = r.dt2; s.local = pp; s.axis = 0; }
  else if (pp < r.dt2 + r.dh2) { s.base = r.T * r.dt2; s.stride = r.dh2; s.local = pp - r.dt2; s.axis = 1; }
  else { s.base = r.T * r.dt2 + r.H * r.dh2; s.stride = r.dh2; s.local = pp - r.dt2 - r.dh2; s.axis = 2; }
  return s;
}

__device__ __forceinline__ int pair_index(const PairSel& s, int t, int h, int w) {
  const int pos = s.axis == 0 ? t : (s.axis == 1 ? h : w);
  return s.base + pos * s.stride + s.local;
}

// (x, y) -> (x cos - y sin, x sin + y cos)
__device__ __forceinline__ float2 rope_rotate(float x, float y, float2 cs) {
  return make_float2(fmaf(x, cs.x, -(y * cs.y)), fmaf(x, cs.y, y * cs.x));
}

// transpose rotation, used for gradients: (x, y) -> (x cos + y sin, -x sin + y cos)
__device__ __forceinline__ float2 rope_rotate_t(float x, float y, float2 cs) {
  return make_float2(fmaf(x, cs.x, y * cs.y), fmaf(y, cs.x, -(x * cs.y)));
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_32b(void* p, uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                              uint32_t w4, uint32_t w5, uint32_t w6, uint32_t w7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "r"(w0), "r"(w1), "r"(w2), "r"(w3), "r"(w4), "r"(w5), "r"(w6), "r"(w7) : "memory");
}

// 64 bytes to global memory: two 32-byte stores when `wide` (dst 32-byte
// aligned), else four 16-byte ones.
__device__ __forceinline__ void st_global_64b(void* dst, const uint32_t (&w)[16], bool wide) {
  if (wide) {
    st_global_32b(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
    st_global_32b(static_cast<uint8_t*>(dst) + 32, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
  } else {
    uint4* d = static_cast<uint4*>(dst);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) d[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
  }
}

// ---------------------------------------------------------------------------
// Shared memory / barriers / bounded waits
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Control block every role of a CTA shares: a CTA-wide abort flag in shared
// memory and the device error word.
struct Ctl {
  volatile int* abort;
  int* err;
};

// Slow path of a bounded wait: give up after kWaitLimitNs, or at once when
// another role already gave up. Records `code` in the error word.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, Ctl c, int code) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (*c.abort) return false;
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *c.abort = 1;
      atomicCAS(c.err, 0, code);
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, Ctl c, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, c, code);
}

// The same waits for barriers that also receive arrivals from the other CTA of
// a cluster (acquire at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
static __device__ __noinline__ bool mbar_wait_cl_slow(uint32_t bar, uint32_t parity, Ctl c, int code) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (*c.abort) return false;
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cl(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *c.abort = 1;
      atomicCAS(c.err, 0, code);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, Ctl c, int code) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  return mbar_wait_cl_slow(bar, parity, c, code);
}
static __device__ __noinline__ void mbar_drain_cl(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cl(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Shared-memory address `addr` of this CTA as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
// Arrive on a barrier of another CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}

// Bounded wait that ignores the abort flag: used only to drain copies and MMAs
// still in flight before a CTA releases its shared memory and TMEM.
static __device__ __noinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" :: "l"((uint64_t)m) : "memory");
}

// Load into this CTA's shared memory, completing on a barrier that may be in
// the other CTA of the pair (`bar` a shared::cluster address from mapa_shared).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
      :: "r"(dst), "l"((uint64_t)m), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// One 128-position tile of a scope: positions p0 .. p0 + 127 of scope s, batch
// b (one 128-row box per 64 channels of a head, 128-byte swizzle). Unpacked:
// through the 5-D scope-gather map over the caller's (B, N, heads, D) tensor
// (dims channel, head, in-group offset, scope, merged (batch, group));
// packed: from the scope-ordered copy (k, B, Lp, heads, D) through a 3-D map
// (channel, head, row), rows past a scope's end holding zeros. The coordinate
// is formed once per tile (its loads sit on the producers' critical path).
struct TileCoord {
  int s;      // scope coordinate of the 5-D map, or -1 for the packed 3-D map
  int row;
};
__device__ __forceinline__ TileCoord scope_tile(const Geom& g, int s, int b, int p0) {
  TileCoord c;
  if (g.packed) {
    c.s = -1;
    c.row = (s * g.B + b) * g.Lp + p0;
  } else {
    c.s = s;
    c.row = b * g.Nn + (p0 >> g.lgG);
  }
  return c;
}
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar, TileCoord c, int c0,
                                          int head) {
  if (c.s < 0) tma_load_3d(dst, m, bar, c0, head, c.row);
  else tma_load_5d(dst, m, bar, c0, head, 0, c.s, c.row);
}

// L2 prefetch of the tile load_tile with the same arguments fetches (no
// shared-memory destination, nothing to wait for): issued a few tiles ahead of
// a work unit's first loads, it turns their HBM latency into an L2 hit.
__device__ __forceinline__ void prefetch_tile(const CUtensorMap* m, TileCoord c, int c0, int head) {
  if (c.s < 0)
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"((uint64_t)m), "r"(c0), "r"(head), "r"(c.row) : "memory");
  else
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];"
                 :: "l"((uint64_t)m), "r"(c0), "r"(head), "r"(0), "r"(c.s), "r"(c.row) : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"((uint64_t)src), "r"(bytes), "r"(bar) : "memory");
}

// Bulk reduce-add of `bytes` fp32 values from shared to global memory (the
// TMA unit adds them element-wise, atomically per element), tracked as a bulk
// group of the issuing thread.
__device__ __forceinline__ void bulk_reduce_add_f32(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
               :: "l"((uint64_t)gdst), "r"(ssrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read their shared source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
// Programmatic dependent launch: a kernel launched by launch_after_previous
// may be scheduled (and run its prologue) while the kernel before it in the
// stream drains; pdl_wait holds it until that kernel has completed and its
// writes are visible. pdl_trigger lets the next kernel be scheduled early.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename Kernel, typename Params>
cudaError_t launch_after_previous(Kernel kernel, int grid, int block, size_t smem, cudaStream_t stream,
                                  const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Wait until every committed bulk group has fully completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Named barrier over `nthreads` threads that ANDs a predicate across them, so a
// group of warps takes the same branch after bounded waits.
template <int ID, int NTHREADS>
__device__ __forceinline__ bool bar_and(bool v) {
  uint32_t out;
  __syncwarp();   // bar.red is the aligned form: the warp must arrive converged
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
               "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(out) : "r"(v ? 1u : 0u), "n"(ID), "n"(NTHREADS) : "memory");
  return out != 0;
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 op this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// CTA-pair (cta_group::2) forms: one M = 256 MMA over the two CTAs' shared
// memory (each CTA holds its 128 rows of A and its half of B's rows, at the
// same offsets) into each CTA's own TMEM, issued by the pair's first CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_pair_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Arrive on the barrier at the same offset in every CTA in `mask` once the
// pair MMAs this thread issued are done.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"(mask) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
               :: "r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// 8-bit operands (kind::f8f6f4, E4M3 A and B, fp32 accumulator): K = 32 per
// instruction, i.e. 32 bytes of a row, the same byte step as kind::f16.
__device__ __forceinline__ void mma8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
               :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
// Instruction descriptor, kind::f8f6f4: E4M3 A and B (format code 0), fp32 D,
// both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Four fp32 values to E4M3 (round to nearest even, saturating at +-448), first
// value in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator.
//  bits 4-5 D type (1 = f32), 7-9 A type (1 = bf16), 10-12 B type (1 = bf16),
//  15 A MN-major, 16 B MN-major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzle.
//  bits 0-13 start >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte
//  offset >> 4, 46-48 = 0b001 (tcgen05 descriptor version), 61-63 = 2 (128B swizzle).
// K-major operands: rows of 64 bf16 (128 B), 8-row groups SBO = 1024 B apart.
// MN-major operands: 64 MN-elements per 128-B row, one row per K index; the
// next 8 K rows are SBO = 1024 B on, the next 64 MN-elements LBO bytes on.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// K-major operand made of row x 64-channel boxes (one per 64 channels, `box`
// bytes apart; 128-row boxes by default): k-step ks of 16 channels starts in
// box ks/4, 32 B into each row.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int ks, uint32_t box = kHalfBytes) {
  return sdesc_sw128(tile + (uint32_t)((ks >> 2) * box + (ks & 3) * 32), 16, 1024);
}

// MN-major operand stored as [K rows][MN columns] in the same boxes: k-step
// ks of 16 rows starts 16 * 128 B further; MN columns 64.. are in the next box.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int ks, uint32_t box = kHalfBytes) {
  return sdesc_sw128(tile + (uint32_t)(ks * 2048), box, 1024);
}

// Descriptor of k-step ks from the k-step-0 descriptor: the start address field
// (bits 0-13, in 16-byte units) advances by the step's byte offset >> 4 (shared
// memory addresses stay below 2^18, so the field never carries).
__device__ __forceinline__ uint64_t kmajor_step(uint64_t d0, int ks, uint32_t box = kHalfBytes) {
  return d0 + (uint64_t)(((ks >> 2) * box + (ks & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t mnmajor_step(uint64_t d0, int ks) { return d0 + (uint64_t)(ks * 128); }

// tcgen05.ld, 32 lanes x 32 bit, 32 consecutive columns; waits for completion.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.st, 32 lanes x 32 bit, 16 consecutive columns (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
         "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// tcgen05.ld, 32 lanes x 32 bit, 16 consecutive columns; waits for completion.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.st, 32 lanes x 32 bit, 16 consecutive columns of floats (no wait).
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float (&v)[16]) {
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
  tmem_st16(taddr, r);
}


// Two tcgen05.ld 32x32b.x16 (16 consecutive columns at each of two addresses), one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float (&a)[16], float (&b)[16]) {
  uint32_t r[16], q[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]),
        "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15])
      : "r"(ta), "r"(tb) : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(q[i]);
  }
}

// tcgen05.ld, 32 lanes x 32 bit, 64 consecutive columns, one wait for all of them.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.ld, 32 lanes x 32 bit, 128 consecutive columns, one wait for all of them.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.st, 32 lanes x 32 bit, 8 consecutive columns (no wait).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Packed two-lane fp32 arithmetic (one instruction for two values).
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  return ((unsigned long long)__float_as_uint(b) << 32) | __float_as_uint(a);
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& a, float& b) {
  a = __uint_as_float((uint32_t)v);
  b = __uint_as_float((uint32_t)(v >> 32));
}
// (a0, a1) * (b0, b1) + (c0, c1), round to nearest
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ unsigned long long fsub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long fmul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Largest of the 128 scores of a softmax row held in registers: four chains of
// three-input maxima. With RAGGED, scores at or past `valid` (keys beyond the
// scope's end in its last tile) are first set to -inf.
template <bool RAGGED>
__device__ __forceinline__ float row_max128(float (&x)[128], int valid) {
  if constexpr (RAGGED) {
#pragma unroll
    for (int e = 0; e < 128; ++e) x[e] = e < valid ? x[e] : -INFINITY;
  }
  float mm[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) mm[i] = fmaxf(x[i], x[i + 4]);
#pragma unroll
  for (int e = 8; e < 128; e += 8) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mm[i] = fmax3(mm[i], x[e + i], x[e + 4 + i]);
  }
  return fmax3(mm[0], mm[1], fmaxf(mm[2], mm[3]));
}

}  // namespace skp
