// Test hooks: the index map and the RoPE rotation exactly as the attention
// kernels compute them (same device functions, same cos/sin table).
#include "skiparse_internal.h"

namespace skp {

// For every token i: (scope, position) from the forward map, cross-checked
// against the inverse map the kernels use to address rows; a mismatch is
// reported as scope -1.
__global__ void skiparse_debug_index_map_kernel(const __grid_constant__ DebugParams p) {
  const Geom& g = p.g;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < g.N; i += gridDim.x * blockDim.x) {
    int s, pos;
    scope_pos_of(g, i, s, pos);
    const bool ok = s >= 0 && s < g.k && pos >= 0 && pos < scope_len(g, s) && token_of(g, s, pos) == i;
    p.scope_of_token[i] = ok ? s : -1;
    p.pos_of_token[i] = pos;
  }
}

// One warp per (b, token, head) row; each lane rotates channel pairs of the
// row with the shared-memory table, as the forward kernel's RoPE warps do.
template <int D>
__global__ void skiparse_debug_rope_kernel(const __grid_constant__ DebugParams p) {
  extern __shared__ float2 tab[];
  rope_build_table(tab, p.rope, threadIdx.x, blockDim.x);
  __syncthreads();
  const Geom& g = p.g;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const long long rows = (long long)g.B * g.N * g.heads;
  for (long long row = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); row < rows; row += (long long)gridDim.x * wpb) {
    int b, i, head;
    row_coords(g, (int)row, b, i, head);
    int t, hh, w;
    token_coords(p.rope, i, t, hh, w);
    for (int pp = lane; pp < D / 2; pp += 32) {
      const PairSel sel = pair_select(p.rope, pp);
      const float2 cs = tab[pair_index(sel, t, hh, w)];
      const uint32_t u = *reinterpret_cast<const uint32_t*>(p.x + (size_t)row * D + 2 * pp);
      const float2 o = rope_rotate(bf16lo(u), bf16hi(u), cs);
      *reinterpret_cast<float2*>(p.x_rot + (size_t)row * D + 2 * pp) = o;
    }
  }
}

// Bounded-wait check: one CTA of two warps, each waiting on its own mbarrier
// that nothing ever arrives at, through the same bounded wait the attention
// kernels use. The first wait to run out records `code` in the error word and
// raises the CTA's abort flag; the other returns as soon as it sees the flag.
// Nothing is left in flight, so the CTA exits normally.
__global__ void skiparse_debug_wait_timeout_kernel(int* err, int code) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  const Ctl c{&abort_flag, err};
  if ((threadIdx.x & 31) == 0) mbar_wait(smem_u32(&bars[threadIdx.x >> 5]), 0, c, code);
  __syncthreads();
}

cudaError_t launch_debug_wait_timeout(int* err, int code, cudaStream_t stream) {
  skiparse_debug_wait_timeout_kernel<<<1, 64, 0, stream>>>(err, code);
  return cudaGetLastError();
}

cudaError_t launch_debug_index_map(const DebugParams& p, cudaStream_t stream) {
  const int grid = (p.g.N + 255) / 256;
  skiparse_debug_index_map_kernel<<<grid > 0 ? grid : 1, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_debug_rope(const DebugParams& p, cudaStream_t stream) {
  const size_t smem = (size_t)p.rope.entries * sizeof(float2);
  const long long rows = (long long)p.g.B * p.g.N * p.g.heads;
  long long grid = (rows + 7) / 8;
  if (grid > 4096) grid = 4096;
  cudaError_t e;
  if (p.g.D == 128) {
    e = cudaFuncSetAttribute(skiparse_debug_rope_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    skiparse_debug_rope_kernel<128><<<(int)grid, 256, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(skiparse_debug_rope_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    skiparse_debug_rope_kernel<64><<<(int)grid, 256, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace skp
