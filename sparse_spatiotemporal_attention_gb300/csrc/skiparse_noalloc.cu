// Allocation-free backward entry point.
//
// Some callers cannot allocate device memory at the point where they need the
// backward pass: code running under a custom allocator that forbids calls back
// into the CUDA allocator, plugins and embedded runtimes that own all device
// memory themselves, or hosts where a stray cudaMalloc would synchronise the
// device or break a pre-planned memory budget. For them this file keeps the
// backward's scratch (fp32 dQ accumulator, rotated q/k, per-scope LSE/delta,
// RoPE table) in one file-scope device array of fixed size, so a call needs
// nothing but the caller's inputs and outputs.
//
// The array lives in this library's device image: every GPU that loads the
// library holds SKIPARSE_NOALLOC_SCRATCH_BYTES of it until the process exits.
#include <mutex>

#include "../../include/skiparse.h"
#include "skiparse_internal.h"

namespace {

constexpr size_t kScratchBytes = SKIPARSE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
void* g_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached. The cache is keyed by the
// device's current context too: after cudaDeviceReset, or under another
// context the caller made current, the library's device image (and the array
// in it) is a different one, so the address is looked up again.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SKIPARSE_ERR_DEVICE;
  }
  void* ctx = skp::current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev] || g_ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SKIPARSE_ERR_DEVICE;
    }
    g_addr[dev] = p;
    g_ctx[dev] = skp::current_context();   // the runtime makes the primary context current if none was
  }
  *out = g_addr[dev];
  return SKIPARSE_OK;
}

}  // namespace

extern "C" int skiparse_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                         int B, int heads, int N, int D, int T, int H, int W,
                                         int sparse_k, int mode, float rope_theta, cudaStream_t stream) {
  const size_t need = skiparse_attn_bwd_workspace_bytes(B, heads, N, D, T, H, W, sparse_k, mode);
  if (need == 0) {
    // invalid or empty sizes: the regular entry point reports them (no scratch is touched)
    return skiparse_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, nullptr, 0, B, heads, N, D, T, H, W,
                             sparse_k, mode, rope_theta, stream);
  }
  if (need > kScratchBytes) return SKIPARSE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != SKIPARSE_OK) return st;
  return skiparse_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, scratch, kScratchBytes, B, heads, N, D, T, H, W,
                           sparse_k, mode, rope_theta, stream);
}
