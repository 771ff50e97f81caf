// Internal interface between the C-ABI host layer and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "skiparse_dev.cuh"

namespace skp {

// Codes written to the device error word when a bounded wait runs out:
// kernel base + barrier index; the backward main kernel adds 0x80.
enum : int {
  ERR_KERNEL_FWD = 0x1000,
  ERR_KERNEL_BWD = 0x2000,
  ERR_KERNEL_PROJ = 0x3000,
  ERR_SMEM_ALIGN = 0x7001,
};

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;   // scope-gather maps over rotated q, rotated k (workspace) and v
  const uint16_t* q;              // pre-RoPE inputs (RoPE pass)
  const uint16_t* k;
  const uint16_t* v;              // v (pack pass)
  uint16_t* qr;                   // workspace: rotated q, bf16 (B, N, heads, D); packed: (k, B, Lp, heads, D)
  uint16_t* kr;                   // workspace: rotated k, likewise
  uint16_t* vr;                   // packed only: v in scope order (k, B, Lp, heads, D)
  int rotate;                     // 0: rope_theta = 0 (q, k arrive rotated; the pack pass only copies)
  float2* rope_gtab;              // workspace: the cos/sin table (written by skiparse_rope_table_kernel)
  Geom g;
  RopeParams rope;
  uint16_t* out;                  // bf16 (B, N, heads, D)
  float* lse;                     // (B, heads, N)
  int* err;                       // device error word
  int n_units;                    // B * heads * k * ceil(n_tiles / 2): pairs of Q tiles
  // Work items: units [0, n_full) whole, then the remaining units each split
  // into `pieces` key-tile ranges whose partial O, m, l go to part_o / part_ml
  // (slot = item - n_full) and are merged by skiparse_fwd_merge_kernel.
  int n_full, pieces, n_items;
  float* part_o;                  // workspace: (slots, 256 rows, D) fp32 unnormalised O of a Q-tile pair
  float2* part_ml;                // workspace: (slots, 256 rows) (m, l) in base 2
  float scale_log2;               // log2(e) / sqrt(D)
};

// Most slots of split units a forward call uses (the pieces of its last round
// of units run together, one per SM).
constexpr int kMaxFwdSlots = 160;

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // maps over rotated q, rotated k, v, dout (128-row boxes)
  Geom g;
  RopeParams rope;
  const uint16_t* q;       // pre-RoPE inputs
  const uint16_t* k;
  const uint16_t* out;
  const uint16_t* dout;
  const float* lse;
  const uint16_t* v;
  uint16_t* qr;            // rotated q, bf16 (B, N, heads, D): workspace, or the forward's;
                           // packed: scope order (k, B, Lp, heads, D)
  uint16_t* kr;            // rotated k, likewise
  uint16_t* vp;            // packed only: v in scope order (workspace, or the forward's)
  uint16_t* dop;           // packed only: dout in scope order (workspace)
  int write_qkv;           // packed only: 1 the pack pass writes qr, kr (rotated) and vp; 0 they are the forward's
  float* dq_acc;           // workspace: fp32 (B, heads, k, Lp, D), scope order
  float* lse2s;            // workspace: lse * log2(e), scope order (B, heads, k, Lp)
  float* delta_s;          // workspace: rowsum(dO * O), scope order (B, heads, k, Lp)
  float2* rope_tab;        // workspace: cos/sin table
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  int* err;
  int n_units;             // B * heads * k * n_tiles (one K/V tile each)
  int rotate_qk;           // 1: the preprocess writes qr / kr from q / k; 0: qr / kr are given
  int Lp;                  // L rounded up to a multiple of 128
  float scale;             // 1 / sqrt(D)
  float scale_log2;        // log2(e) / sqrt(D)
};

struct Fwd8Params {
  CUtensorMap tm_q8, tm_k8;       // 8-bit q / k codes, scope-tile order (Lp rows per scope): E4M3 (128 bytes
                                  // per row, 128 x 128 boxes) or INT8 held as bf16 (128 channels per row,
                                  // 64-channel x 128-row boxes)
  CUtensorMap tm_vt;              // 8-bit V^T per scope: (Lp keys, 128 channels, scopes), 128 x 128 boxes
  CUtensorMap tm_q, tm_k;         // bf16 inputs q / k through the scope gather (prep kernel's staged tiles)
  Geom g;
  RopeParams rope;
  const uint16_t* q;              // bf16 (B, N, heads, D) inputs
  const uint16_t* k;
  const uint16_t* v;
  float2* rope_gtab;              // workspace: the cos/sin table (written by skiparse_rope_table_kernel)
  uint8_t* q8;                    // workspace: codes (scopes, Lp, 128), scope order, 1 or 2 bytes each
  uint8_t* k8;
  uint8_t* vt8;                   // workspace: E4M3 V^T (scopes, 128, Lp)
  float* sq;                      // workspace: q scale per scope-order row (scopes, Lp)
  float* sk;                      // workspace: k scale per K tile (scopes, n_tiles)
  unsigned* vmax;                 // workspace: max |v| per (b, head, channel) as float bits
  uint16_t* out;                  // bf16 (B, N, heads, D)
  float* lse;                     // (B, heads, N)
  int* err;
  int n_units;                    // scopes * ceil(n_tiles / 2)
  int Lp;                         // L rounded up to a multiple of 128
  int prep_stages;                // prep kernel's q / k staging ring: 1 or 2 tiles
  float scale_log2;               // log2(e) / sqrt(D)
};

// Q/K/V projection with the RoPE epilogue: [q | k | v] = x W^T (+ bias), RoPE on q and k.
struct ProjParams {
  CUtensorMap tm_x;               // x bf16 (M rows, C channels): boxes of 64 channels x 128 rows
  CUtensorMap tm_w;               // W bf16 (3 heads D rows, C channels): boxes of 64 channels x BN rows
  RopeParams rope;
  const uint16_t* bias;           // bf16 [3 heads D] or nullptr
  uint16_t* q;                    // bf16 (B, N, heads, D) outputs
  uint16_t* k;
  uint16_t* v;
  int* err;
  FastDiv fN;                     // row -> token
  int M, C, hd, D;                // rows B N, channels, heads D, head dim
  int m_tiles, n_tiles;           // 128-row tiles, BN-column tiles
  int k_steps;                    // ceil(C / channels per stage)
  int stages;                     // pipeline depth (2 .. 4)
  int stage_off;                  // byte offset of stage 0 in shared memory (1024-aligned)
};

struct DebugParams {
  Geom g;
  RopeParams rope;
  const uint16_t* x;
  float* x_rot;
  int* scope_of_token;
  int* pos_of_token;
};

// The calling thread's current CUDA context (driver handle), or nullptr. Device
// variables of this library have one copy per context, so addresses looked up
// with cudaGetSymbolAddress are cached per (device, context).
void* current_context();

// Grid-stride row kernels: at most one wave of resident CTAs (SMs x CTAs per SM
// at this block size and shared memory), so no partial second wave idles SMs.
template <typename K>
inline int one_wave(K kernel, int grid, int threads, size_t smem, int sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1) {
    cudaGetLastError();
    return grid;
  }
  const long long wave = (long long)per_sm * sms;
  return grid < wave ? grid : (int)wave;
}

// Shared-memory bytes and launch helpers (defined next to each kernel).
size_t fwd_smem_bytes(int D);
size_t fwd_rope_smem_bytes(int rope_entries);
int fwd_units(const Geom& g);
cudaError_t launch_fwd_rope(const FwdParams& p, int grid, int sms, cudaStream_t stream);
cudaError_t launch_fwd_pack(const FwdParams& p, int grid, int sms, cudaStream_t stream);
cudaError_t launch_fwd(const FwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_fwd_merge(const FwdParams& p, int sms, cudaStream_t stream);
// the 3D RoPE cos/sin table of `r` into tab (r.entries float2), once per call
cudaError_t launch_rope_table(const RopeParams& r, float2* tab, cudaStream_t stream);

// si8: the mixed recipe (INT8 q / k codes held as bf16 for S, E4M3 P and v)
size_t fwd8_smem_bytes(bool si8);
size_t fwd8_qk_row_bytes(bool si8);
// prep kernel: shared memory for a staging ring of `stages` q / k tiles, and the
// ring size to launch with: 1 when two such CTAs fit on an SM (`smem_sm` bytes,
// 1 KB reserved per CTA), else the largest (2, 1) that fits one CTA (`optin`
// bytes); 0 when none does
int fwd8_prep_stages(int T, int H, int W, size_t optin, size_t smem_sm);
int fwd8_units(const Geom& g);
cudaError_t launch_fwd8_vmax(const Fwd8Params& p, cudaStream_t stream);
cudaError_t launch_fwd8_prep(const Fwd8Params& p, bool si8, int sms, cudaStream_t stream);
cudaError_t launch_fwd8(const Fwd8Params& p, bool si8, int grid, cudaStream_t stream);

int proj_bn(int hd);
size_t proj_stage_bytes(int bn);
int proj_stage_channels();
size_t proj_header_bytes(int rope_entries);
cudaError_t launch_proj(const ProjParams& p, int bn, int grid, cudaStream_t stream);

size_t bwd_main_smem_bytes(int D);
cudaError_t launch_bwd_pre(const BwdParams& p, int grid, int sms, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_post(const BwdParams& p, int grid, int sms, cudaStream_t stream);

cudaError_t launch_debug_index_map(const DebugParams& p, cudaStream_t stream);
cudaError_t launch_debug_rope(const DebugParams& p, cudaStream_t stream);
cudaError_t launch_debug_wait_timeout(int* err, int code, cudaStream_t stream);

}  // namespace skp
