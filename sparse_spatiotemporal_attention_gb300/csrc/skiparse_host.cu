// C-ABI host layer: argument validation, TMA tensor maps that fold the
// Skiparse rearrange into strides, kernel launches, device error word, tracing.
//
// The scope gather ("Open-Sora Plan" docs, "Skiparse Attention", single and
// group skip rearrange patterns) becomes a 5-D tensor map over the caller's
// (B, N, heads, D) buffer. With G = 1 (single) or G = k (group), token
// i = n*k*G + s*G + kk, so the token axis splits into (n, s, kk); n and b merge
// because b's stride is exactly N/(k*G) times n's:
//   dim 0  channel d         extent D            stride 2 B
//   dim 1  head              extent heads        stride D*2
//   dim 2  kk (in-group)     extent G            stride heads*D*2
//   dim 3  s (scope)         extent k            stride G*heads*D*2
//   dim 4  (b, n) merged     extent B*N/(k*G)    stride k*G*heads*D*2
// A box of (64, 1, G, 1, 128/G) elements is 128 consecutive positions of one
// scope (position p = n*G + kk), landing as 128 rows of 128 B with 128-byte
// swizzle. Rows past the end of a scope read the next batch's rows or zero
// fill; the kernels mask them.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/skiparse.h"
#include "skiparse_internal.h"

using namespace skp;

__device__ int g_skiparse_error_word;

namespace skp {

void* current_context() {
  typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

}  // namespace skp

namespace {

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  bool ready = false;
  void* ctx = nullptr;  // the context the cached error-word address belongs to
  int sms = 0;
  int smem_optin = 0;
  int smem_sm = 0;     // shared memory per SM (all resident CTAs)
  int cc = 0;
  int* err_word = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

// Current device's facts; SKIPARSE_ERR_DEVICE if there is none or it is not sm_103.
int device_info(DeviceInfo& out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SKIPARSE_ERR_DEVICE;
  }
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  // a new context on this device (a reset, or a caller's own context) holds
  // its own copy of the library's device variables: look their address up again
  if (d.ready && d.ctx != ctx) d.ready = false;
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
      cudaGetLastError();
      return SKIPARSE_ERR_DEVICE;
    }
    d.cc = major * 10 + minor;
    void* addr = nullptr;
    if (d.cc == 103) {
      if (cudaGetSymbolAddress(&addr, g_skiparse_error_word) != cudaSuccess) {
        cudaGetLastError();
        return SKIPARSE_ERR_DEVICE;
      }
    }
    d.err_word = static_cast<int*>(addr);
    d.ctx = current_context();   // the runtime makes the primary context current if none was
    d.ready = true;
  }
  if (d.cc != 103) return SKIPARSE_ERR_DEVICE;
  out = d;
  return SKIPARSE_OK;
}

// ---------------------------------------------------------------- tracing

struct TraceRec {
  int id;
  cudaEvent_t a, b;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;

template <class F>
cudaError_t traced_launch(int id, cudaStream_t stream, F&& launch) {
  bool on;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    on = g_trace_on;
  }
  if (!on) return launch();
  TraceRec r{id, nullptr, nullptr};
  if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return cudaGetLastError();
  cudaEventRecord(r.a, stream);
  const cudaError_t e = launch();
  cudaEventRecord(r.b, stream);
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.push_back(r);
  return e;
}

// ---------------------------------------------------------------- validation

struct Shape {
  int B, heads, N, D, T, H, W, k, mode;
  bool empty;
  long long elems;     // B*N*heads*D
  int rope_entries;
};

int check_shape(int B, int heads, int N, int D, int T, int H, int W, int k, int mode, float theta, Shape& s) {
  if (mode != SKIPARSE_SINGLE && mode != SKIPARSE_GROUP) return SKIPARSE_ERR_INVALID_ARG;
  if (B < 0 || heads < 0 || N < 0 || T < 0 || H < 0 || W < 0 || k < 1 || D < 0) return SKIPARSE_ERR_INVALID_ARG;
  if (!(theta >= 0.0f) || !std::isfinite(theta)) return SKIPARSE_ERR_INVALID_ARG;   // 0: no rotation
  if ((long long)T * H * W != (long long)N) return SKIPARSE_ERR_SHAPE;
  s = Shape{B, heads, N, D, T, H, W, k, mode, false, 0, 0};
  if (B == 0 || heads == 0 || N == 0) {
    s.empty = true;
    return SKIPARSE_OK;
  }
  if (D != 64 && D != 128) return SKIPARSE_ERR_UNSUPPORTED;
  // any N: scopes of unequal length when k (single) or k^2 (group) does not divide it
  if (mode == SKIPARSE_GROUP && 128 % k != 0) return SKIPARSE_ERR_UNSUPPORTED;
  const long long entries = (long long)T * (D / 8) + (long long)H * (3 * D / 16) + (long long)W * (3 * D / 16);
  if (entries > kMaxRopeEntries) return SKIPARSE_ERR_UNSUPPORTED;
  s.rope_entries = (int)entries;
  s.elems = (long long)B * N * heads * D;
  const long long G = mode == SKIPARSE_SINGLE ? 1 : k;
  const long long L0 = (N / (k * G)) * G + std::min<long long>(N % (k * G), G);   // scope 0, the longest
  const long long tiles = (L0 + kTile - 1) / kTile;
  const long long units = (long long)B * heads * k * tiles;
  const long long packed_rows = (long long)k * B * tiles * kTile * heads;         // scope-ordered copies
  if (s.elems > (1ll << 46) || units >= (1ll << 31) || (long long)B * N * heads >= (1ll << 31) ||
      packed_rows >= (1ll << 31))
    return SKIPARSE_ERR_UNSUPPORTED;
  return SKIPARSE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  const void* p;
  size_t bytes;
};

bool overlaps(const Range& a, const Range& b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a.bytes && b.bytes && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// outputs must not overlap inputs or each other
bool any_alias(const std::vector<Range>& outs, const std::vector<Range>& ins) {
  for (size_t i = 0; i < outs.size(); ++i) {
    for (const Range& r : ins)
      if (overlaps(outs[i], r)) return true;
    for (size_t j = i + 1; j < outs.size(); ++j)
      if (overlaps(outs[i], outs[j])) return true;
  }
  return false;
}

Geom make_geom(const Shape& s) {
  Geom g;
  g.B = s.B;
  g.heads = s.heads;
  g.N = s.N;
  g.D = s.D;
  g.k = s.k;
  g.G = s.mode == SKIPARSE_SINGLE ? 1 : s.k;
  g.lgG = 0;
  while ((1 << g.lgG) < g.G) ++g.lgG;
  g.fk = make_fastdiv(s.k);
  g.fkG = make_fastdiv(s.k * g.G);
  g.fheads = make_fastdiv(s.heads > 0 ? s.heads : 1);
  g.fN = make_fastdiv(s.N > 0 ? s.N : 1);
  g.fB = make_fastdiv(s.B > 0 ? s.B : 1);
  g.Qb = s.N / (s.k * g.G);
  g.Rb = s.N % (s.k * g.G);
  g.L = scope_len(g, 0);
  g.Nn = g.L / g.G;
  g.n_tiles = (g.L + kTile - 1) / kTile;
  g.Lp = g.n_tiles * kTile;
  g.fLp = make_fastdiv(g.Lp > 0 ? g.Lp : 1);
  // scopes of unequal length are read from scope-ordered copies: the gather
  // maps' per-dimension bounds cannot stop a read past the end of a shorter scope
  g.packed = g.Rb != 0 ? 1 : 0;
  g.s0 = 0;
  g.sstep = 1;
  g.ks = s.k;
  return g;
}

// Restricts a geometry to the scopes first, first + step, ... below k.
int set_subset(Geom& g, int first, int step) {
  if (first < 0 || step < 1) return SKIPARSE_ERR_INVALID_ARG;
  g.s0 = first;
  g.sstep = step;
  g.ks = first < g.k ? (g.k - 1 - first) / step + 1 : 0;
  return SKIPARSE_OK;
}

RopeParams make_rope(const Shape& s, float theta) {
  RopeParams r;
  std::memset(&r, 0, sizeof(r));
  const int dt = s.D / 4, dh = 3 * s.D / 8;
  r.T = s.T;
  r.H = s.H;
  r.W = s.W;
  r.dt2 = dt / 2;
  r.dh2 = dh / 2;
  r.entries = s.rope_entries;
  r.fHW = make_fastdiv(s.H * s.W > 0 ? s.H * s.W : 1);
  r.fW = make_fastdiv(s.W > 0 ? s.W : 1);
  // rope_theta == 0 means q and k arrive rotated: every angle is 0 (cos 1, sin 0),
  // which makes each rotation an exact identity
  for (int j = 0; j < r.dt2; ++j) r.om_t[j] = theta == 0.0f ? 0.0 : std::pow((double)theta, -2.0 * j / dt);
  for (int j = 0; j < r.dh2; ++j) r.om_hw[j] = theta == 0.0f ? 0.0 : std::pow((double)theta, -2.0 * j / dh);
  return r;
}

bool encode_scope_map(CUtensorMap* m, const void* base, const Geom& g) {
  const int box_rows = kTile;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t row = (cuuint64_t)g.heads * g.D * 2;
  const cuuint64_t dims[5] = {(cuuint64_t)g.D, (cuuint64_t)g.heads, (cuuint64_t)g.G, (cuuint64_t)g.k,
                              (cuuint64_t)g.B * g.Nn};
  const cuuint64_t strides[4] = {(cuuint64_t)g.D * 2, row, row * g.G, row * g.G * g.k};
  if (box_rows % g.G != 0) return false;
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)g.G, 1, (cuuint32_t)(box_rows / g.G)};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// 3-D bf16 map over a scope-ordered copy (k, B, Lp, heads, D): dims (channel,
// head, row), a box of 64 channels x 1 head x 128 rows with 128-byte swizzle.
bool encode_packed_map(CUtensorMap* m, const void* base, const Geom& g) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)g.D, (cuuint64_t)g.heads, (cuuint64_t)g.k * g.B * g.Lp};
  const cuuint64_t strides[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.heads * g.D * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bytes of one scope-ordered bf16 copy (k, B, Lp, heads, D)
size_t packed_bytes(const Geom& g) { return (size_t)g.k * g.B * g.Lp * g.heads * g.D * 2; }

// Partial results of the split units of a forward's last round: O (256 rows x
// D fp32) and (m, l) per row for each slot.
// at most kMaxFwdSlots, and never more than the call's (unit, K tile) pairs
size_t fwd_part_slots(const Shape& s) {
  const Geom g = make_geom(s);
  const long long pairs = (long long)s.B * s.heads * s.k * ((g.n_tiles + 1) / 2) * g.n_tiles;
  return (size_t)std::min<long long>(kMaxFwdSlots, pairs);
}
size_t fwd_part_o_bytes(const Shape& s) { return align256(fwd_part_slots(s) * 256 * s.D * 4); }
size_t fwd_part_ml_bytes(const Shape& s) { return align256(fwd_part_slots(s) * 256 * sizeof(float2)); }

// Forward workspace: rotated q and k in row order, or (unequal scopes) q, k
// and v in scope order; then the split units' partial results.
size_t fwd_copies_bytes(const Shape& s) {
  const Geom g = make_geom(s);
  if (g.packed) return 3 * align256(packed_bytes(g));
  return 2 * align256((size_t)s.elems * 2);
}
size_t rope_tab_bytes() { return align256((size_t)kMaxRopeEntries * sizeof(float2)); }
size_t fwd_ws_bytes(const Shape& s) {
  return fwd_copies_bytes(s) + fwd_part_o_bytes(s) + fwd_part_ml_bytes(s) + rope_tab_bytes();
}
// offset of the cos/sin table in the forward workspace (its last region)
size_t fwd_tab_offset(const Shape& s) { return fwd_ws_bytes(s) - rope_tab_bytes(); }

// How a forward's units spread over the SMs: whole units in full rounds, and
// the last round's units split into key ranges when that round leaves at least
// half of the SMs idle (every piece then runs at once, one per SM).
void plan_fwd_items(FwdParams& p, int sms, int slots) {
  const int U = p.n_units;
  const int rounds = (U + sms - 1) / sms;
  const int R = U - (rounds - 1) * sms;             // units of the last round, 1 .. sms
  int pieces = std::min(std::min(sms / R, slots / R), p.g.n_tiles);
  if (pieces < 2) {
    p.n_full = U;
    p.pieces = 1;
    p.n_items = U;
    return;
  }
  p.n_full = U - R;
  p.pieces = pieces;
  p.n_items = p.n_full + R * pieces;
}

// 2-D bf16 tensor map over a row-major (rows, cols) matrix: boxes of 64 columns
// (128 bytes, 128-byte swizzle) x box_rows rows; reads past either edge fill zeros.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D byte tensor map, 128 x 128-byte boxes with 128-byte swizzle: dims
// (d0 innermost, d1, d2), byte strides s1, s2.
bool encode_bytes_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                     uint64_t s2) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map, 64-element x 128-row boxes with 128-byte swizzle: dims
// (d0 innermost, d1, d2), byte strides s1, s2; reads past an edge fill zeros.
bool encode_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 8-bit forward workspace: q, k codes (scopes, Lp, 128) (E4M3 bytes, or INT8
// codes as bf16 for the mixed recipe) and E4M3 V^T (scopes, 128, Lp), q scales
// per scope-order row, k scales per K tile, max |v| per (b, head, channel),
// the cos/sin table; for scopes of unequal length, scope-ordered bf16 copies
// of q, k and v (the prep kernel's tile loads read q and k from them).
struct Ws8Layout {
  size_t q8, k8, vt8, sq, sk, vmax, tab, copies, total;
  int Lp, scopes;
};

Ws8Layout ws8_layout(const Shape& s, bool si8) {
  Ws8Layout w;
  w.Lp = make_geom(s).Lp;
  w.scopes = s.B * s.heads * s.k;
  const size_t rows = (size_t)w.scopes * w.Lp;
  const size_t qk_row = fwd8_qk_row_bytes(si8);
  size_t off = 0;
  w.q8 = off;   off += align256(rows * qk_row);
  w.k8 = off;   off += align256(rows * qk_row);
  w.vt8 = off;  off += align256(rows * 128);
  w.sq = off;   off += align256(rows * 4);
  w.sk = off;   off += align256((size_t)w.scopes * (w.Lp / kTile) * 4);
  w.vmax = off; off += align256((size_t)s.B * s.heads * 128 * 4);
  w.tab = off;  off += align256((size_t)kMaxRopeEntries * sizeof(float2));
  const Geom g = make_geom(s);
  w.copies = off; off += g.packed ? 3 * align256(packed_bytes(g)) : 0;
  w.total = off;
  return w;
}

struct WsLayout {
  size_t dq_acc, qr, kr, vp, dop, lse2s, delta_s, tab, total;
  int Lp;
};

// with_qk = false: the rotated q / k come from the forward pass's workspace and
// their regions are left out (the full layout is a superset).
// Scopes of unequal length (packed): q, k (rotated) and v in scope order unless
// the forward's are reused (with_qk = false), and dout in scope order.
WsLayout ws_layout(const Shape& s, bool with_qk = true) {
  WsLayout w;
  const size_t e = (size_t)s.elems;
  const Geom g = make_geom(s);
  w.Lp = g.Lp;
  const size_t stats = (size_t)s.B * s.heads * s.k * w.Lp;
  const size_t copy = g.packed ? align256(packed_bytes(g)) : align256(e * 2);
  size_t off = 0;
  w.dq_acc = off; off += align256(stats * (size_t)s.D * 4);   // scope order (B, heads, k, Lp, D)
  w.qr = off;     off += with_qk ? copy : 0;
  w.kr = off;     off += with_qk ? copy : 0;
  w.vp = off;     off += (g.packed && with_qk) ? copy : 0;
  w.dop = off;    off += g.packed ? copy : 0;
  w.lse2s = off;  off += align256(stats * 4);
  w.delta_s = off; off += align256(stats * 4);
  w.tab = off;    off += align256((size_t)s.rope_entries * sizeof(float2));
  w.total = off;
  return w;
}

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) return SKIPARSE_OK;
  cudaGetLastError();
  return SKIPARSE_ERR_LAUNCH;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================

extern "C" {

const char* skiparse_status_string(int status) {
  switch (status) {
    case SKIPARSE_OK: return "ok";
    case SKIPARSE_ERR_INVALID_ARG: return "invalid argument (NULL pointer, negative size, bad mode or rope_theta)";
    case SKIPARSE_ERR_SHAPE: return "shape mismatch (N != T*H*W; the 8-bit forwards also need k (single) / k*k (group) to divide N)";
    case SKIPARSE_ERR_UNSUPPORTED: return "unsupported configuration (D must be 64 or 128; group k must divide 128; RoPE table too large)";
    case SKIPARSE_ERR_ALIGNMENT: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case SKIPARSE_ERR_DEVICE: return "no CUDA device, or the current device is not sm_103 (GB300)";
    case SKIPARSE_ERR_WORKSPACE: return "workspace missing or too small";
    case SKIPARSE_ERR_LAUNCH: return "tensor-map encode or kernel launch failed";
    case SKIPARSE_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (see detail code)";
    case SKIPARSE_ERR_ALIAS: return "an output overlaps an input or another output";
    default: return "unknown status";
  }
}

const char* skiparse_kernel_name(int id) {
  switch (id) {
    case 0: return "skiparse_fwd_kernel";
    case 1: return "skiparse_bwd_pre_kernel";
    case 2: return "skiparse_bwd_main_kernel";
    case 3: return "skiparse_bwd_post_kernel";
    case 4: return "skiparse_fwd_rope_kernel";
    case 5: return "skiparse_fwd8_vmax_kernel";
    case 6: return "skiparse_fwd8_prep_kernel";
    case 7: return "skiparse_fwd8_kernel";
    case 8: return "skiparse_qkv_rope_kernel";
    case 9: return "skiparse_fwdm8_prep_kernel";
    case 10: return "skiparse_fwdm8_kernel";
    case 11: return "skiparse_fwd_merge_kernel";
    default: return "unknown";
  }
}

size_t skiparse_attn_fwd_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W, int sparse_k, int mode) {
  Shape s;
  if (check_shape(B, heads, N, D, T, H, W, sparse_k, mode, 10000.0f, s) != SKIPARSE_OK || s.empty) return 0;
  return fwd_ws_bytes(s);
}

}  // extern "C"

namespace {

// Forward over the scopes first, first + step, ... (all of them for 0, 1).
int fwd_impl(const void* q, const void* k, const void* v, void* out, float* lse, void* workspace,
             size_t workspace_bytes, int B, int heads, int N, int D, int T, int H, int W, int sparse_k, int mode,
             float rope_theta, int scope_first, int scope_step, cudaStream_t stream) {
  Shape s;
  int st = check_shape(B, heads, N, D, T, H, W, sparse_k, mode, rope_theta, s);
  if (st != SKIPARSE_OK || s.empty) return st;
  Geom geom = make_geom(s);
  if ((st = set_subset(geom, scope_first, scope_step)) != SKIPARSE_OK) return st;
  if (geom.ks == 0) return SKIPARSE_OK;
  if (!q || !k || !v || !out || !lse) return SKIPARSE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return SKIPARSE_ERR_ALIGNMENT;
  const size_t need = fwd_ws_bytes(s);
  if (!workspace || workspace_bytes < need) return SKIPARSE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SKIPARSE_ERR_ALIGNMENT;
  const size_t tb = (size_t)s.elems * 2, lb = (size_t)B * heads * N * 4;
  if (any_alias({{out, tb}, {lse, lb}, {workspace, need}}, {{q, tb}, {k, tb}, {v, tb}})) return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = device_info(dev)) != SKIPARSE_OK) return st;
  if ((size_t)dev.smem_optin < fwd_smem_bytes(D) || (size_t)dev.smem_optin < fwd_rope_smem_bytes(s.rope_entries))
    return SKIPARSE_ERR_UNSUPPORTED;

  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = geom;
  p.rope = make_rope(s, rope_theta);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  const bool rotate = rope_theta != 0.0f;            // 0: q and k are already rotated
  p.rotate = rotate ? 1 : 0;
  if (p.g.packed) {
    // scopes of unequal length: q, k (rotated) and v in scope order
    const size_t pb = align256(packed_bytes(p.g));
    p.qr = reinterpret_cast<uint16_t*>(ws);
    p.kr = reinterpret_cast<uint16_t*>(ws + pb);
    p.vr = reinterpret_cast<uint16_t*>(ws + 2 * pb);
    if (!encode_packed_map(&p.tm_q, p.qr, p.g) || !encode_packed_map(&p.tm_k, p.kr, p.g) ||
        !encode_packed_map(&p.tm_v, p.vr, p.g))
      return SKIPARSE_ERR_LAUNCH;
  } else {
    const size_t half = align256((size_t)s.elems * 2);
    p.qr = reinterpret_cast<uint16_t*>(ws);
    p.kr = reinterpret_cast<uint16_t*>(ws + half);
    if (!encode_scope_map(&p.tm_q, rotate ? p.qr : q, p.g) || !encode_scope_map(&p.tm_k, rotate ? p.kr : k, p.g) ||
        !encode_scope_map(&p.tm_v, v, p.g))
      return SKIPARSE_ERR_LAUNCH;
  }
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = dev.err_word;
  p.n_units = fwd_units(p.g);
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  plan_fwd_items(p, dev.sms, (int)fwd_part_slots(s));
  p.part_o = reinterpret_cast<float*>(ws + fwd_copies_bytes(s));
  p.part_ml = reinterpret_cast<float2*>(ws + fwd_copies_bytes(s) + fwd_part_o_bytes(s));
  p.rope_gtab = reinterpret_cast<float2*>(ws + fwd_tab_offset(s));
  const long long rows = (long long)B * N * heads;
  long long rgrid = (rows + 15) / 16;                 // 8 warps per CTA, 2 rows per warp
  if (rgrid > 8ll * dev.sms) rgrid = 8ll * dev.sms;
  const int grid = p.n_items < dev.sms ? p.n_items : dev.sms;
  if (p.g.packed || rotate) {
    st = launch_status(launch_rope_table(p.rope, p.rope_gtab, stream));
    if (st != SKIPARSE_OK) return st;
  }
  if (p.g.packed) {
    st = launch_status(traced_launch(4, stream, [&] { return launch_fwd_pack(p, 8 * dev.sms, dev.sms, stream); }));
    if (st != SKIPARSE_OK) return st;
  } else if (rotate) {
    st = launch_status(traced_launch(4, stream, [&] { return launch_fwd_rope(p, (int)rgrid, dev.sms, stream); }));
    if (st != SKIPARSE_OK) return st;
  }
  st = launch_status(traced_launch(0, stream, [&] { return launch_fwd(p, grid, stream); }));
  if (st != SKIPARSE_OK || p.n_items == p.n_full) return st;
  return launch_status(traced_launch(11, stream, [&] { return launch_fwd_merge(p, dev.sms, stream); }));
}

}  // namespace

extern "C" {

int skiparse_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      void* workspace, size_t workspace_bytes,
                      int B, int heads, int N, int D, int T, int H, int W,
                      int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  return fwd_impl(q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode, rope_theta,
                  0, 1, stream);
}

int skiparse_attn_fwd_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                             void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                             cudaStream_t stream) {
  return fwd_impl(q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode, rope_theta,
                  scope_first, scope_step, stream);
}

size_t skiparse_attn_fwd_fp8_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W, int sparse_k,
                                             int mode) {
  Shape s;
  if (check_shape(B, heads, N, D, T, H, W, sparse_k, mode, 10000.0f, s) != SKIPARSE_OK || s.empty || D != 128) return 0;
  return ws8_layout(s, false).total;
}

size_t skiparse_attn_fwd_mixed8_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W, int sparse_k,
                                                int mode) {
  Shape s;
  if (check_shape(B, heads, N, D, T, H, W, sparse_k, mode, 10000.0f, s) != SKIPARSE_OK || s.empty || D != 128) return 0;
  return ws8_layout(s, true).total;
}

}  // extern "C"

namespace {

// The 8-bit forward: si8 = false all-E4M3 operands, si8 = true INT8 q / k for S;
// the scopes scope_first, scope_first + scope_step, ... (0, 1: all).
int fwd8_impl(bool si8, const void* q, const void* k, const void* v, void* out, float* lse, void* workspace,
              size_t workspace_bytes, int B, int heads, int N, int D, int T, int H, int W, int sparse_k, int mode,
              float rope_theta, int scope_first, int scope_step, cudaStream_t stream) {
  Shape s;
  int st = check_shape(B, heads, N, D, T, H, W, sparse_k, mode, rope_theta, s);
  if (st != SKIPARSE_OK || s.empty) return st;
  if (D != 128) return SKIPARSE_ERR_UNSUPPORTED;
  Geom geom = make_geom(s);
  if ((st = set_subset(geom, scope_first, scope_step)) != SKIPARSE_OK) return st;
  if (geom.ks == 0) return SKIPARSE_OK;
  if (!q || !k || !v || !out || !lse) return SKIPARSE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return SKIPARSE_ERR_ALIGNMENT;
  const Ws8Layout w = ws8_layout(s, si8);
  if (!workspace || workspace_bytes < w.total) return SKIPARSE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SKIPARSE_ERR_ALIGNMENT;
  const size_t tb = (size_t)s.elems * 2, lb = (size_t)B * heads * N * 4;
  if (any_alias({{out, tb}, {lse, lb}, {workspace, w.total}}, {{q, tb}, {k, tb}, {v, tb}})) return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = device_info(dev)) != SKIPARSE_OK) return st;
  const int prep_stages = fwd8_prep_stages(s.T, s.H, s.W, (size_t)dev.smem_optin, (size_t)dev.smem_sm);
  if ((size_t)dev.smem_optin < fwd8_smem_bytes(si8) || prep_stages == 0) return SKIPARSE_ERR_UNSUPPORTED;

  Fwd8Params p;
  std::memset(&p, 0, sizeof(p));
  p.g = geom;
  p.rope = make_rope(s, rope_theta);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.q8 = ws + w.q8;
  p.k8 = ws + w.k8;
  p.vt8 = ws + w.vt8;
  p.sq = reinterpret_cast<float*>(ws + w.sq);
  p.sk = reinterpret_cast<float*>(ws + w.sk);
  p.vmax = reinterpret_cast<unsigned*>(ws + w.vmax);
  p.rope_gtab = reinterpret_cast<float2*>(ws + w.tab);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = dev.err_word;
  p.Lp = w.Lp;
  p.prep_stages = prep_stages;
  p.n_units = fwd8_units(p.g);
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  const uint64_t Lp = (uint64_t)w.Lp, sc = (uint64_t)w.scopes;
  const bool qk_ok = si8 ? encode_bf16_3d(&p.tm_q8, p.q8, 128, Lp, sc, 256, 256 * Lp) &&
                               encode_bf16_3d(&p.tm_k8, p.k8, 128, Lp, sc, 256, 256 * Lp)
                         : encode_bytes_3d(&p.tm_q8, p.q8, 128, Lp, sc, 128, 128 * Lp) &&
                               encode_bytes_3d(&p.tm_k8, p.k8, 128, Lp, sc, 128, 128 * Lp);
  // q and k tiles for the prep kernel: through the scope gather, or (unequal
  // scopes, which no gather map can bound) from scope-ordered copies that the
  // pack pass writes, unrotated (the prep kernel applies RoPE itself)
  FwdParams pk;
  std::memset(&pk, 0, sizeof(pk));
  if (p.g.packed) {
    const size_t pb = align256(packed_bytes(p.g));
    pk.g = p.g;
    pk.rope = p.rope;
    pk.q = p.q;
    pk.k = p.k;
    pk.v = p.v;
    pk.qr = reinterpret_cast<uint16_t*>(ws + w.copies);
    pk.kr = reinterpret_cast<uint16_t*>(ws + w.copies + pb);
    pk.vr = reinterpret_cast<uint16_t*>(ws + w.copies + 2 * pb);
    pk.rotate = 0;
    pk.err = dev.err_word;
  }
  const bool maps_ok = p.g.packed ? encode_packed_map(&p.tm_q, pk.qr, p.g) && encode_packed_map(&p.tm_k, pk.kr, p.g)
                                  : encode_scope_map(&p.tm_q, q, p.g) && encode_scope_map(&p.tm_k, k, p.g);
  if (!qk_ok || !encode_bytes_3d(&p.tm_vt, p.vt8, Lp, 128, sc, Lp, 128 * Lp) || !maps_ok) return SKIPARSE_ERR_LAUNCH;
  const int grid = p.n_units < dev.sms ? p.n_units : dev.sms;
  if (cudaMemsetAsync(p.vmax, 0, (size_t)B * heads * 128 * 4, stream) != cudaSuccess) return launch_status(cudaErrorUnknown);
  st = launch_status(traced_launch(5, stream, [&] { return launch_fwd8_vmax(p, stream); }));
  if (st != SKIPARSE_OK) return st;
  if (p.g.packed) {
    st = launch_status(traced_launch(4, stream, [&] { return launch_fwd_pack(pk, 8 * dev.sms, dev.sms, stream); }));
    if (st != SKIPARSE_OK) return st;
  }
  st = launch_status(launch_rope_table(p.rope, p.rope_gtab, stream));
  if (st != SKIPARSE_OK) return st;
  st = launch_status(traced_launch(si8 ? 9 : 6, stream, [&] { return launch_fwd8_prep(p, si8, dev.sms, stream); }));
  if (st != SKIPARSE_OK) return st;
  return launch_status(traced_launch(si8 ? 10 : 7, stream, [&] { return launch_fwd8(p, si8, grid, stream); }));
}

}  // namespace

extern "C" {

int skiparse_attn_fwd_fp8(const void* q, const void* k, const void* v, void* out, float* lse,
                          void* workspace, size_t workspace_bytes,
                          int B, int heads, int N, int D, int T, int H, int W,
                          int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  return fwd8_impl(false, q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode,
                   rope_theta, 0, 1, stream);
}

int skiparse_attn_fwd_mixed8(const void* q, const void* k, const void* v, void* out, float* lse,
                             void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  return fwd8_impl(true, q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode,
                   rope_theta, 0, 1, stream);
}

int skiparse_attn_fwd_fp8_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes,
                                 int B, int heads, int N, int D, int T, int H, int W,
                                 int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                                 cudaStream_t stream) {
  return fwd8_impl(false, q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode,
                   rope_theta, scope_first, scope_step, stream);
}

int skiparse_attn_fwd_mixed8_scopes(const void* q, const void* k, const void* v, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes,
                                    int B, int heads, int N, int D, int T, int H, int W,
                                    int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                                    cudaStream_t stream) {
  return fwd8_impl(true, q, k, v, out, lse, workspace, workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode,
                   rope_theta, scope_first, scope_step, stream);
}

size_t skiparse_attn_bwd_workspace_bytes(int B, int heads, int N, int D, int T, int H, int W, int sparse_k, int mode) {
  Shape s;
  if (check_shape(B, heads, N, D, T, H, W, sparse_k, mode, 10000.0f, s) != SKIPARSE_OK || s.empty) return 0;
  return ws_layout(s).total;
}

}  // extern "C"

namespace {

// Backward: q / k given (rotated here; fwd_ws == nullptr), or the forward
// pass's workspace (q == k == nullptr) holding its rotated q / k (row order), or
// for scopes of unequal length its scope-ordered q, k and v.
int bwd_impl(const void* q, const void* k, const void* fwd_ws, size_t fwd_ws_given,
             const void* v, const void* out, const float* lse, const void* dout, void* dq, void* dk, void* dv,
             void* workspace, size_t workspace_bytes, int B, int heads, int N, int D, int T, int H, int W,
             int sparse_k, int mode, float rope_theta, int scope_first, int scope_step, cudaStream_t stream) {
  Shape s;
  int st = check_shape(B, heads, N, D, T, H, W, sparse_k, mode, rope_theta, s);
  if (st != SKIPARSE_OK || s.empty) return st;
  Geom geom = make_geom(s);
  if ((st = set_subset(geom, scope_first, scope_step)) != SKIPARSE_OK) return st;
  if (geom.ks == 0) return SKIPARSE_OK;
  const bool saved = fwd_ws != nullptr;
  const bool rotate = rope_theta != 0.0f;            // 0: q and k are already rotated
  if (saved && !rotate) return SKIPARSE_ERR_INVALID_ARG;   // the forward wrote no rotated copies
  if (!v || !out || !lse || !dout || !dq || !dk || !dv) return SKIPARSE_ERR_INVALID_ARG;
  if (!saved && (!q || !k)) return SKIPARSE_ERR_INVALID_ARG;
  const size_t tb = (size_t)s.elems * 2, lb = (size_t)B * heads * N * 4;
  const size_t fwd_need = fwd_ws_bytes(s);
  const uint8_t* fw = static_cast<const uint8_t*>(fwd_ws);
  const size_t fcopy = geom.packed ? align256(packed_bytes(geom)) : align256(tb);
  const void* qa = saved ? fw : q;
  const void* ka = saved ? fw + fcopy : k;
  if (!aligned16(qa) || !aligned16(ka) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return SKIPARSE_ERR_ALIGNMENT;
  const WsLayout w = ws_layout(s, !saved && (rotate || geom.packed));
  if (!workspace || workspace_bytes < w.total) return SKIPARSE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SKIPARSE_ERR_ALIGNMENT;
  if (saved && fwd_ws_given < fwd_need) return SKIPARSE_ERR_WORKSPACE;
  std::vector<Range> ins = {{v, tb}, {out, tb}, {lse, lb}, {dout, tb}};
  if (saved) ins.push_back({fwd_ws, fwd_need});
  else {
    ins.push_back({q, tb});
    ins.push_back({k, tb});
  }
  if (any_alias({{dq, tb}, {dk, tb}, {dv, tb}, {workspace, w.total}}, ins)) return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = device_info(dev)) != SKIPARSE_OK) return st;
  if ((size_t)dev.smem_optin < bwd_main_smem_bytes(D)) return SKIPARSE_ERR_UNSUPPORTED;

  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = geom;
  p.rope = make_rope(s, rope_theta);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.out = static_cast<const uint16_t*>(out);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
  p.lse2s = reinterpret_cast<float*>(ws + w.lse2s);
  p.delta_s = reinterpret_cast<float*>(ws + w.delta_s);
  // the cos/sin table: the forward call's when its workspace is reused (same
  // sizes and rope_theta), else built here into this workspace
  p.rope_tab = saved ? reinterpret_cast<float2*>(const_cast<uint8_t*>(fw) + fwd_tab_offset(s))
                     : reinterpret_cast<float2*>(ws + w.tab);
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.err = dev.err_word;
  p.Lp = w.Lp;
  p.n_units = B * heads * p.g.ks * p.g.n_tiles;
  p.scale = (float)(1.0 / std::sqrt((double)D));
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  bool maps_ok;
  if (p.g.packed) {
    // scopes of unequal length: every operand from a scope-ordered copy
    p.write_qkv = saved ? 0 : 1;
    p.rotate_qk = rotate ? 1 : 0;
    uint8_t* fwm = const_cast<uint8_t*>(fw);
    p.qr = reinterpret_cast<uint16_t*>(saved ? fwm : ws + w.qr);
    p.kr = reinterpret_cast<uint16_t*>(saved ? fwm + fcopy : ws + w.kr);
    p.vp = reinterpret_cast<uint16_t*>(saved ? fwm + 2 * fcopy : ws + w.vp);
    p.dop = reinterpret_cast<uint16_t*>(ws + w.dop);
    maps_ok = encode_packed_map(&p.tm_q, p.qr, p.g) && encode_packed_map(&p.tm_k, p.kr, p.g) &&
              encode_packed_map(&p.tm_v, p.vp, p.g) && encode_packed_map(&p.tm_do, p.dop, p.g);
  } else {
    p.rotate_qk = (!saved && rotate) ? 1 : 0;
    p.qr = saved ? const_cast<uint16_t*>(static_cast<const uint16_t*>(qa))
                 : rotate ? reinterpret_cast<uint16_t*>(ws + w.qr) : const_cast<uint16_t*>(static_cast<const uint16_t*>(q));
    p.kr = saved ? const_cast<uint16_t*>(static_cast<const uint16_t*>(ka))
                 : rotate ? reinterpret_cast<uint16_t*>(ws + w.kr) : const_cast<uint16_t*>(static_cast<const uint16_t*>(k));
    maps_ok = encode_scope_map(&p.tm_q, p.qr, p.g) && encode_scope_map(&p.tm_k, p.kr, p.g) &&
              encode_scope_map(&p.tm_v, v, p.g) && encode_scope_map(&p.tm_do, dout, p.g);
  }
  if (!maps_ok) return SKIPARSE_ERR_LAUNCH;

  const long long rows = (long long)B * N * heads;
  long long rgrid = (rows + 15) / 16;                 // 8 warps per CTA, 2 rows per warp
  if (rgrid > 8ll * dev.sms) rgrid = 8ll * dev.sms;
  const int pregrid = p.g.packed ? 8 * dev.sms : (int)rgrid;
  const int mgrid = p.n_units < dev.sms ? p.n_units : dev.sms;
  if (!saved) {
    st = launch_status(launch_rope_table(p.rope, p.rope_tab, stream));
    if (st != SKIPARSE_OK) return st;
  }
  st = launch_status(traced_launch(1, stream, [&] { return launch_bwd_pre(p, pregrid, dev.sms, stream); }));
  if (st != SKIPARSE_OK) return st;
  st = launch_status(traced_launch(2, stream, [&] { return launch_bwd_main(p, mgrid, stream); }));
  if (st != SKIPARSE_OK) return st;
  return launch_status(traced_launch(3, stream, [&] { return launch_bwd_post(p, (int)rgrid, dev.sms, stream); }));
}

}  // namespace

extern "C" {

int skiparse_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                      int B, int heads, int N, int D, int T, int H, int W,
                      int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  return bwd_impl(q, k, nullptr, 0, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, heads, N, D, T, H,
                  W, sparse_k, mode, rope_theta, 0, 1, stream);
}

int skiparse_attn_bwd_scopes(const void* q, const void* k, const void* v, const void* out, const float* lse,
                             const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int heads, int N, int D, int T, int H, int W,
                             int sparse_k, int mode, float rope_theta, int scope_first, int scope_step,
                             cudaStream_t stream) {
  return bwd_impl(q, k, nullptr, 0, v, out, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, heads, N, D, T, H,
                  W, sparse_k, mode, rope_theta, scope_first, scope_step, stream);
}

int skiparse_attn_bwd_saved(const void* fwd_workspace, size_t fwd_workspace_bytes, const void* v, const void* out,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, int B, int heads, int N, int D, int T, int H, int W,
                            int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  Shape s;
  const int st = check_shape(B, heads, N, D, T, H, W, sparse_k, mode, rope_theta, s);
  if (st != SKIPARSE_OK || s.empty) return st;
  if (!fwd_workspace) return SKIPARSE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(fwd_workspace) & 255u) != 0) return SKIPARSE_ERR_ALIGNMENT;
  // the forward workspace holds rotated q, then rotated k (and, for scopes of
  // unequal length, v), each 256-byte aligned
  return bwd_impl(nullptr, nullptr, fwd_workspace, fwd_workspace_bytes, v, out, lse, dout, dq, dk, dv, workspace,
                  workspace_bytes, B, heads, N, D, T, H, W, sparse_k, mode, rope_theta, 0, 1, stream);
}

int skiparse_debug_index_map(int* scope_of_token, int* pos_of_token, int N, int sparse_k, int mode,
                             cudaStream_t stream) {
  if (mode != SKIPARSE_SINGLE && mode != SKIPARSE_GROUP) return SKIPARSE_ERR_INVALID_ARG;
  if (N < 0 || sparse_k < 1) return SKIPARSE_ERR_INVALID_ARG;
  if (N == 0) return SKIPARSE_OK;
  if (!scope_of_token || !pos_of_token) return SKIPARSE_ERR_INVALID_ARG;
  if (mode == SKIPARSE_GROUP && 128 % sparse_k != 0) return SKIPARSE_ERR_UNSUPPORTED;
  if (any_alias({{scope_of_token, (size_t)N * 4}, {pos_of_token, (size_t)N * 4}}, {})) return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  int st = device_info(dev);
  if (st != SKIPARSE_OK) return st;
  DebugParams p;
  std::memset(&p, 0, sizeof(p));
  Shape s{1, 1, N, 64, 1, 1, N, sparse_k, mode, false, 0, 0};
  p.g = make_geom(s);
  p.scope_of_token = scope_of_token;
  p.pos_of_token = pos_of_token;
  return launch_status(launch_debug_index_map(p, stream));
}

int skiparse_debug_rope(const void* x, float* x_rot, int B, int heads, int N, int D, int T, int H, int W,
                        float rope_theta, cudaStream_t stream) {
  Shape s;
  int st = check_shape(B, heads, N, D, T, H, W, 1, SKIPARSE_SINGLE, rope_theta, s);
  if (st != SKIPARSE_OK || s.empty) return st;
  if (!x || !x_rot) return SKIPARSE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_rot)) return SKIPARSE_ERR_ALIGNMENT;
  if (any_alias({{x_rot, (size_t)s.elems * 4}}, {{x, (size_t)s.elems * 2}})) return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  if ((st = device_info(dev)) != SKIPARSE_OK) return st;
  DebugParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = make_geom(s);
  p.rope = make_rope(s, rope_theta);
  p.x = static_cast<const uint16_t*>(x);
  p.x_rot = x_rot;
  return launch_status(launch_debug_rope(p, stream));
}

int skiparse_debug_wait_timeout(int code, cudaStream_t stream) {
  if (code <= 0) return SKIPARSE_ERR_INVALID_ARG;
  DeviceInfo dev;
  int st = device_info(dev);
  if (st != SKIPARSE_OK) return st;
  return launch_status(launch_debug_wait_timeout(dev.err_word, code, stream));
}

int skiparse_qkv_rope(const void* x, const void* w, const void* bias, void* q, void* k, void* v, int B, int N,
                      int C, int heads, int D, int T, int H, int W, float rope_theta, cudaStream_t stream) {
  if (B < 0 || N < 0 || C < 0 || heads < 0 || D < 0 || T < 0 || H < 0 || W < 0) return SKIPARSE_ERR_INVALID_ARG;
  if (!(rope_theta >= 0.0f) || !std::isfinite(rope_theta)) return SKIPARSE_ERR_INVALID_ARG;   // 0: no rotation
  if ((long long)T * H * W != (long long)N) return SKIPARSE_ERR_SHAPE;
  if (B == 0 || N == 0 || heads == 0) return SKIPARSE_OK;
  if (D != 64 && D != 128) return SKIPARSE_ERR_UNSUPPORTED;
  const long long hd = (long long)heads * D;
  if (C < 8 || C % 8 != 0 || hd % 128 != 0) return SKIPARSE_ERR_UNSUPPORTED;
  const long long entries = (long long)T * (D / 8) + (long long)H * (3 * D / 16) + (long long)W * (3 * D / 16);
  if (entries > kMaxRopeEntries) return SKIPARSE_ERR_UNSUPPORTED;
  const long long M = (long long)B * N;
  if (M >= (1ll << 31) || 3 * hd >= (1ll << 31) || M * hd > (1ll << 46) || M * C > (1ll << 46))
    return SKIPARSE_ERR_UNSUPPORTED;
  if (!x || !w || !q || !k || !v) return SKIPARSE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      (bias && !aligned16(bias)))
    return SKIPARSE_ERR_ALIGNMENT;
  const size_t out_bytes = (size_t)(M * hd) * 2;
  if (any_alias({{q, out_bytes}, {k, out_bytes}, {v, out_bytes}},
                {{x, (size_t)(M * C) * 2}, {w, (size_t)(3 * hd * C) * 2}, {bias, bias ? (size_t)(3 * hd) * 2 : 0}}))
    return SKIPARSE_ERR_ALIAS;
  DeviceInfo dev;
  int st = device_info(dev);
  if (st != SKIPARSE_OK) return st;
  const int bn = proj_bn((int)hd);
  const size_t header = proj_header_bytes((int)entries);
  const size_t per_stage = proj_stage_bytes(bn);
  long long stages = ((long long)dev.smem_optin - (long long)header) / (long long)per_stage;
  if (stages > 6) stages = 6;
  if (stages < 2) return SKIPARSE_ERR_UNSUPPORTED;
  Shape s{B, heads, N, D, T, H, W, 1, SKIPARSE_SINGLE, false, M * hd, (int)entries};
  ProjParams p;
  std::memset(&p, 0, sizeof(p));
  p.rope = make_rope(s, rope_theta);
  p.bias = static_cast<const uint16_t*>(bias);
  p.q = static_cast<uint16_t*>(q);
  p.k = static_cast<uint16_t*>(k);
  p.v = static_cast<uint16_t*>(v);
  p.err = dev.err_word;
  p.fN = make_fastdiv(N);
  p.M = (int)M;
  p.C = C;
  p.hd = (int)hd;
  p.D = D;
  p.m_tiles = (int)((M + 127) / 128);
  p.n_tiles = (int)(3 * hd / bn);
  p.k_steps = (C + proj_stage_channels() - 1) / proj_stage_channels();
  p.stages = (int)stages;
  p.stage_off = (int)header;
  if (!encode_bf16_2d(&p.tm_x, x, (uint64_t)C, (uint64_t)M, 128) ||
      !encode_bf16_2d(&p.tm_w, w, (uint64_t)C, (uint64_t)(3 * hd), (uint32_t)bn / 2))
    return SKIPARSE_ERR_LAUNCH;
  // clusters of two CTAs, one per vertically adjacent pair of tiles
  const long long pairs = (long long)((p.m_tiles + 1) / 2) * p.n_tiles;
  const long long clusters = pairs < dev.sms / 2 ? pairs : dev.sms / 2;
  const int grid = (int)(2 * clusters);
  return launch_status(traced_launch(8, stream, [&] { return launch_proj(p, bn, grid, stream); }));
}

int skiparse_device_error(int* detail) {
  DeviceInfo dev;
  int st = device_info(dev);
  if (st != SKIPARSE_OK) return st;
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return SKIPARSE_ERR_LAUNCH;
  }
  if (cudaMemcpyFromSymbol(&v, g_skiparse_error_word, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return SKIPARSE_ERR_LAUNCH;
  }
  const int zero = 0;
  cudaMemcpyToSymbol(g_skiparse_error_word, &zero, sizeof(int));
  if (detail) *detail = v;
  return v == 0 ? SKIPARSE_OK : SKIPARSE_ERR_DEVICE_TIMEOUT;
}

int skiparse_trace_begin(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = true;
  return SKIPARSE_OK;
}

int skiparse_trace_end(float* ms_per_kernel, int* launches_per_kernel, int n) {
  std::vector<TraceRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    g_trace_on = false;
    recs.swap(g_trace);
  }
  for (int i = 0; i < n; ++i) {
    if (ms_per_kernel) ms_per_kernel[i] = 0.f;
    if (launches_per_kernel) launches_per_kernel[i] = 0;
  }
  int st = SKIPARSE_OK;
  for (const TraceRec& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      cudaGetLastError();
      st = SKIPARSE_ERR_LAUNCH;
    }
    if (r.id >= 0 && r.id < n) {
      if (ms_per_kernel) ms_per_kernel[r.id] += ms;
      if (launches_per_kernel) launches_per_kernel[r.id] += 1;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  return st;
}

}  // extern "C"
