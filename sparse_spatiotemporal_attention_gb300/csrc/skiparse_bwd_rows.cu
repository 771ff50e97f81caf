// Skiparse attention backward, row kernels: the preprocess before and the
// post pass after the main kernel (skiparse_bwd.cu). Both are HBM-bound, one
// warp per (b, token, head) row of the original layout.
//
//  preprocess  delta = rowsum(dO * O) and lse * log2(e) at the row's
//              scope-order slot, rotated bf16 copies of q and k (so the main
//              loop reloads no RoPE), the row's dQ~ accumulator zeroed, and
//              the cos/sin table written to the workspace (for the main
//              kernel's dK epilogue and the post pass).
//  post        dq = R^T (scale * dQ~_acc) -> bf16 at the original row.
#include "skiparse_internal.h"

namespace skp {

// ===========================================================================
// preprocess and post: one warp per (b, token, head) row
// ===========================================================================

constexpr int kRowThreads = 256;

// 8-byte (PPL = 2) or 4-byte (PPL = 1) slice of a bf16 row owned by one lane.
template <int PPL>
__device__ __forceinline__ void ld_slice(const uint16_t* src, uint32_t (&v)[PPL]) {
  if (PPL == 2) {
    const uint2 a = *reinterpret_cast<const uint2*>(src);
    v[0] = a.x;
    v[PPL - 1] = a.y;
  } else {
    v[0] = *reinterpret_cast<const uint32_t*>(src);
  }
}
template <int PPL>
__device__ __forceinline__ void st_slice(uint16_t* dst, const uint32_t (&v)[PPL]) {
  if (PPL == 2) *reinterpret_cast<uint2*>(dst) = make_uint2(v[0], v[PPL - 1]);
  else *reinterpret_cast<uint32_t*>(dst) = v[0];
}

// Preprocess: per (b, token, head) row, delta = rowsum(dO * O) and lse * log2(e)
// at the row's scope-order slot and the row's dQ accumulator zeroed; with ROT,
// also rotated bf16 copies of q and k (without it the forward pass's copies are
// reused). One warp per row, R rows per iteration so each lane has the loads
// of all R rows in flight before it uses any.
template <int D, bool ROT, bool SUBSET>
__global__ void __launch_bounds__(kRowThreads, ROT ? 5 : 8) skiparse_bwd_pre_kernel(const __grid_constant__ BwdParams p) {
  constexpr int R = 2;
  extern __shared__ float2 tab[];
  const Geom& g = p.g;
  // the table (built once per call in the workspace) rotates q and k here
  if (ROT) {
    rope_load_table(tab, p.rope_tab, p.rope.entries, threadIdx.x, blockDim.x);
    __syncthreads();
  }
  constexpr int PPL = D / 64;               // channel pairs per lane
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  PairSel sel[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) sel[e] = pair_select(p.rope, lane * PPL + e);
  const long long rows = (long long)g.B * g.N * g.heads;
  const long long stride = (long long)gridDim.x * wpb;
  for (long long r0 = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); r0 < rows; r0 += R * stride) {
    uint32_t qv[R][PPL], kv[R][PPL], ov[R][PPL], dv[R][PPL];
    float lse[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      lse[u] = 0.f;
      const long long row = r0 + u * stride;
      if (row >= rows) continue;
      const size_t base = (size_t)row * D + lane * 2 * PPL;
      if (ROT) {
        ld_slice<PPL>(p.q + base, qv[u]);
        ld_slice<PPL>(p.k + base, kv[u]);
      }
      ld_slice<PPL>(p.out + base, ov[u]);
      ld_slice<PPL>(p.dout + base, dv[u]);
      if (lane == 0) {
        int b, i, head;
        row_coords(g, (int)row, b, i, head);
        lse[u] = p.lse[((size_t)b * g.heads + head) * g.N + i];
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const long long row = r0 + u * stride;
      if (row >= rows) continue;
      int b, i, head;
      row_coords(g, (int)row, b, i, head);
      if (SUBSET) {                                  // only the scopes this call computes
        int s, pp;
        scope_pos_of(g, i, s, pp);
        if (!in_subset(g, s)) continue;
      }
      float dsum = 0.f;
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        dsum = fmaf(bf16lo(ov[u][e]), bf16lo(dv[u][e]), dsum);
        dsum = fmaf(bf16hi(ov[u][e]), bf16hi(dv[u][e]), dsum);
      }
      const size_t base = (size_t)row * D + lane * 2 * PPL;
      if (ROT) {
        int t, hh, w;
        token_coords(p.rope, i, t, hh, w);
        uint32_t qo[PPL], ko[PPL];
#pragma unroll
        for (int e = 0; e < PPL; ++e) {
          const float2 cs = tab[pair_index(sel[e], t, hh, w)];
          const float2 a = rope_rotate(bf16lo(qv[u][e]), bf16hi(qv[u][e]), cs);
          const float2 c = rope_rotate(bf16lo(kv[u][e]), bf16hi(kv[u][e]), cs);
          qo[e] = pack_bf16(a.x, a.y);
          ko[e] = pack_bf16(c.x, c.y);
        }
        st_slice<PPL>(p.qr + base, qo);
        st_slice<PPL>(p.kr + base, ko);
      }
      int s, pp;
      scope_pos_of(g, i, s, pp);
      const size_t idx = (((size_t)b * g.heads + head) * g.k + s) * p.Lp + pp;   // scope-order row
      float* acc = p.dq_acc + idx * D + lane * 2 * PPL;
      if (PPL == 2) *reinterpret_cast<float4*>(acc) = make_float4(0.f, 0.f, 0.f, 0.f);
      else *reinterpret_cast<float2*>(acc) = make_float2(0.f, 0.f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      if (lane == 0) {
        p.delta_s[idx] = dsum;
        p.lse2s[idx] = lse[u] * 1.4426950408889634f;
      }
    }
  }
}

// Preprocess for scopes of unequal length (N not divisible by k or k^2): the
// same per-row work in scope order, one warp per row (s, b, pos, head) of the
// scope-ordered copies (k, B, Lp, heads, D), head fastest. A row inside its
// scope gathers its token's dO (and, with write_qkv, q and k, rotated, and v)
// into the copies; a row past the scope's end writes zeros there, so the main
// kernel's MMAs never meet uninitialised padding. delta and lse * log2(e) go to
// the scope-order slot, whose dQ~ accumulator row is zeroed.
template <int D>
__global__ void __launch_bounds__(kRowThreads) skiparse_bwd_pack_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ float2 tab[];
  const Geom& g = p.g;
  rope_load_table(tab, p.rope_tab, p.rope.entries, threadIdx.x, blockDim.x);
  __syncthreads();
  constexpr int PPL = D / 64;
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  PairSel sel[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) sel[e] = pair_select(p.rope, lane * PPL + e);
  const bool rot = p.rotate_qk != 0;
  const long long rows = (long long)g.k * g.B * g.Lp * g.heads;
  const long long stride = (long long)gridDim.x * wpb;
  for (long long row = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); row < rows; row += stride) {
    const int sbp = fdiv((int)row, g.fheads);                 // (s * B + b) * Lp + pos
    const int head = (int)row - sbp * g.heads;
    const int sb = fdiv(sbp, g.fLp);
    const int pos = sbp - sb * g.Lp;
    const int s = fdiv(sb, g.fB);
    const int b = sb - s * g.B;
    if (!in_subset(g, s)) continue;                  // only the scopes this call computes
    const bool inside = pos < scope_len(g, s);
    uint32_t qv[PPL], kv[PPL], vv[PPL], ov[PPL], dv[PPL];
#pragma unroll
    for (int e = 0; e < PPL; ++e) qv[e] = kv[e] = vv[e] = ov[e] = dv[e] = 0u;
    float lse = 0.f, dsum = 0.f;
    int tok = 0;
    if (inside) {
      tok = token_of(g, s, pos);
      const size_t src = (((size_t)b * g.N + tok) * g.heads + head) * D + lane * 2 * PPL;
      ld_slice<PPL>(p.out + src, ov);
      ld_slice<PPL>(p.dout + src, dv);
      if (p.write_qkv) {
        ld_slice<PPL>(p.q + src, qv);
        ld_slice<PPL>(p.k + src, kv);
        ld_slice<PPL>(p.v + src, vv);
      }
      if (lane == 0) lse = p.lse[((size_t)b * g.heads + head) * g.N + tok];
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        dsum = fmaf(bf16lo(ov[e]), bf16lo(dv[e]), dsum);
        dsum = fmaf(bf16hi(ov[e]), bf16hi(dv[e]), dsum);
      }
      if (p.write_qkv && rot) {
        int t, hh, w;
        token_coords(p.rope, tok, t, hh, w);
#pragma unroll
        for (int e = 0; e < PPL; ++e) {
          const float2 cs = tab[pair_index(sel[e], t, hh, w)];
          const float2 a = rope_rotate(bf16lo(qv[e]), bf16hi(qv[e]), cs);
          const float2 c = rope_rotate(bf16lo(kv[e]), bf16hi(kv[e]), cs);
          qv[e] = pack_bf16(a.x, a.y);
          kv[e] = pack_bf16(c.x, c.y);
        }
      }
    }
    const size_t dst = (size_t)row * D + lane * 2 * PPL;
    st_slice<PPL>(p.dop + dst, dv);
    if (p.write_qkv) {
      st_slice<PPL>(p.qr + dst, qv);
      st_slice<PPL>(p.kr + dst, kv);
      st_slice<PPL>(p.vp + dst, vv);
    }
    const size_t idx = (((size_t)b * g.heads + head) * g.k + s) * p.Lp + pos;   // scope-order slot
    float* acc = p.dq_acc + idx * D + lane * 2 * PPL;
    if (PPL == 2) *reinterpret_cast<float4*>(acc) = make_float4(0.f, 0.f, 0.f, 0.f);
    else *reinterpret_cast<float2*>(acc) = make_float2(0.f, 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    if (lane == 0) {
      p.delta_s[idx] = dsum;
      p.lse2s[idx] = lse * 1.4426950408889634f;
    }
  }
}

// Post: dq = R^T (scale * dQ~) for each (b, token, head) row, read from the
// row's scope-order accumulator slot; four rows per warp iteration.
template <int D, bool SUBSET>
__global__ void __launch_bounds__(kRowThreads) skiparse_bwd_post_kernel(const __grid_constant__ BwdParams p) {
  const Geom& g = p.g;
  constexpr int PPL = D / 64;
  const int lane = threadIdx.x & 31;
  const long long wpb = blockDim.x >> 5;
  PairSel sel[PPL];
#pragma unroll
  for (int e = 0; e < PPL; ++e) sel[e] = pair_select(p.rope, lane * PPL + e);
  const long long rows = (long long)g.B * g.N * g.heads;
  const long long stride = (long long)gridDim.x * wpb;
  constexpr int R = 4;
  for (long long r0 = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); r0 < rows; r0 += R * stride) {
    float x[R][2 * PPL];
    int tt[R], th[R], tw[R];
    bool skip[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const long long row = r0 + u * stride;
      skip[u] = row >= rows;
      if (skip[u]) continue;
      int b, i, head;
      row_coords(g, (int)row, b, i, head);
      int s, pp;
      scope_pos_of(g, i, s, pp);
      if (SUBSET) {
        skip[u] = !in_subset(g, s);                  // dq rows of other scopes stay untouched
        if (skip[u]) continue;
      }
      token_coords(p.rope, i, tt[u], th[u], tw[u]);
      const float* acc = p.dq_acc + ((((size_t)b * g.heads + head) * g.k + s) * p.Lp + pp) * D + lane * 2 * PPL;
      if (PPL == 2) {
        const float4 a = *reinterpret_cast<const float4*>(acc);
        x[u][0] = a.x; x[u][1] = a.y; x[u][2 * PPL - 2] = a.z; x[u][2 * PPL - 1] = a.w;
      } else {
        const float2 a = *reinterpret_cast<const float2*>(acc);
        x[u][0] = a.x; x[u][1] = a.y;
      }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const long long row = r0 + u * stride;
      if (skip[u]) continue;
      uint32_t o[PPL];
#pragma unroll
      for (int e = 0; e < PPL; ++e) {
        const float2 cs = __ldg(&p.rope_tab[pair_index(sel[e], tt[u], th[u], tw[u])]);
        const float2 r = rope_rotate_t(x[u][2 * e] * p.scale, x[u][2 * e + 1] * p.scale, cs);
        o[e] = pack_bf16(r.x, r.y);
      }
      st_slice<PPL>(p.dq + (size_t)row * D + lane * 2 * PPL, o);
    }
  }
}

template <int D, bool ROT>
static cudaError_t launch_pre_variant(const BwdParams& p, int grid, int sms, size_t smem, cudaStream_t stream) {
  auto kernel = p.g.ks < p.g.k ? skiparse_bwd_pre_kernel<D, ROT, true> : skiparse_bwd_pre_kernel<D, ROT, false>;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  grid = one_wave(kernel, grid, kRowThreads, smem, sms);
  kernel<<<grid, kRowThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_pack_variant(const BwdParams& p, int grid, int sms, size_t smem, cudaStream_t stream) {
  const cudaError_t e =
      cudaFuncSetAttribute(skiparse_bwd_pack_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  grid = one_wave(skiparse_bwd_pack_kernel<D>, grid, kRowThreads, smem, sms);
  skiparse_bwd_pack_kernel<D><<<grid, kRowThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdParams& p, int grid, int sms, cudaStream_t stream) {
  const size_t smem = (p.g.packed || p.rotate_qk) ? (size_t)p.rope.entries * sizeof(float2) : 0;
  if (p.g.packed)
    return p.g.D == 128 ? launch_pack_variant<128>(p, grid, sms, smem, stream)
                        : launch_pack_variant<64>(p, grid, sms, smem, stream);
  if (p.g.D == 128)
    return p.rotate_qk ? launch_pre_variant<128, true>(p, grid, sms, smem, stream)
                       : launch_pre_variant<128, false>(p, grid, sms, smem, stream);
  return p.rotate_qk ? launch_pre_variant<64, true>(p, grid, sms, smem, stream)
                     : launch_pre_variant<64, false>(p, grid, sms, smem, stream);
}

cudaError_t launch_bwd_post(const BwdParams& p, int grid, int sms, cudaStream_t stream) {
  const bool sub = p.g.ks < p.g.k;
  auto kernel = p.g.D == 128 ? (sub ? skiparse_bwd_post_kernel<128, true> : skiparse_bwd_post_kernel<128, false>)
                             : (sub ? skiparse_bwd_post_kernel<64, true> : skiparse_bwd_post_kernel<64, false>);
  grid = one_wave(kernel, grid, kRowThreads, 0, sms);
  kernel<<<grid, kRowThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace skp
