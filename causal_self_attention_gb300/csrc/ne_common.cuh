// ne_common.cuh -- shared definitions of the attention kernels: tile sizes,
// launch parameter blocks, and the device-side status codes.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ne {

// Tile geometry: 128 query rows x 128 key columns, head dimension 64 (one
// 128-byte bf16 row per token and head, exactly one 128-byte swizzle atom).
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kHD = 64;
constexpr int kTileBytes = kBM * kHD * 2;  // 16 KiB: one 128 x 64 bf16 tile

// Device status word values (ne_attn_get_device_status maps them to ne_status).
constexpr int NE_DEV_OK = 0;
constexpr int NE_DEV_BAD_SEQLEN = 1;        // a sequence longer than max_seqlen, or
                                            // cu_seqlens outside [0, n_tot]
constexpr int NE_DEV_TIMEOUT_BASE = 0x100;  // + wait site id

// RoPE table: for position p and frequency i < 32, rope[p * 32 + i] = (cos, sin)
// of p * theta_i in fp32, each the fp32 rounding of the double value.
struct RopeTable {
  const float2* cs;   // row layout: cs[p * 32 + i] = (cos, sin) of p * theta_i
  const float4* csw;  // the same values warp-interleaved: for the 32 positions
                      // p = 32 g + l, csw[(16 g + c) * 32 + l] = (cos, sin, cos,
                      // sin) of dims 2c, 2c + 1 of position p, so that a warp
                      // reading 32 consecutive positions reads whole lines
  int capacity;       // number of positions (a multiple of 32)
};

// One attention problem in the packed form: tokens are rows of [N_tot, H, 64];
// sequence s spans rows cu[s] .. cu[s+1]-1.  A fixed-length batch [B, T, H, 64]
// is the packed form with cu = {0, T, 2T, ...}, given implicitly (cu == nullptr).
struct Problem {
  const int* cu_seqlens;  // device, nseq + 1 entries, or nullptr for fixed length
  int nseq;               // B for fixed length
  int max_len;            // T for fixed length; max_seqlen for varlen
  int H;
  int n_tot;              // total rows
  int lse_fixed;          // 1: LSE is [B, H, T]; 0: LSE is [H, N_tot]
};

struct FwdParams {
  Problem pb;
  void* out;         // bf16 or fp32 [N_tot, H, 64]
  int out_f32;
  float* lse;
  float scale_log2;  // softmax scale * log2(e)
  RopeTable rope;
  int* status;
  int rotate_k;      // 1: K tiles are loaded un-rotated and rotated in smem;
                     // 0: the keys come pre-rotated (k')
  int rotate_q;      // 1: Q tiles are rotated in smem; 0: the caller passed q'
  const int* compact = nullptr;  // packed batch: the non-empty items (dealt_item), or nullptr
};

struct BwdParams {
  Problem pb;
  const __nv_bfloat16* q;   // un-rotated inputs, read by the preprocess
  const __nv_bfloat16* k;
  __nv_bfloat16* qr;        // [N_tot, H, 64] bf16 workspace: q' = R(m) q
  __nv_bfloat16* kr;        // [N_tot, H, 64] bf16 workspace: k' = R(n) k
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* delta;     // [H, N_tot] fp32 workspace: D_m = dO_m . O_m
  float* dq_acc;    // [N_tot, H, 64] fp32 workspace (rotated-frame dQ', unscaled)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float scale;
  float scale_log2;
  RopeTable rope;
  int* status;
  int rotate_in;   // 1: the preprocess writes q' = R(m) q, k' = R(n) k into the
                   // workspace; 0: q, k are q', k' already (the caller's)
  int rotate_out;  // 1: the postprocess returns dq = R(m)^T dq', dk = R(n)^T dk';
                   // 0: the gradients w.r.t. q', k' themselves
  const int* sched = nullptr;  // work schedule of the persistent main kernel, or
  int sched_ctas = 0;          // nullptr for the snake order; the grid it was made for
  const int* compact = nullptr;  // packed batch: the non-empty units (dealt_item), or nullptr
};

// Sequence bounds of sequence s.  Returns false (and raises the device status)
// if cu_seqlens puts the sequence outside [0, n_tot] or makes it longer than
// max_len; the caller then skips the sequence.
__device__ __forceinline__ bool seq_bounds(const Problem& pb, int s, int& start, int& len,
                                           int* status) {
  if (pb.cu_seqlens) {
    start = __ldg(pb.cu_seqlens + s);
    const int end = __ldg(pb.cu_seqlens + s + 1);
    len = end - start;
    if (start < 0 || end > pb.n_tot || len < 0 || len > pb.max_len) {
      if (status) atomicCAS(status, 0, NE_DEV_BAD_SEQLEN);
      return false;
    }
  } else {
    start = s * pb.max_len;
    len = pb.max_len;
  }
  return true;
}

// Work dealing of the persistent kernels: the index r (in the longest-first
// order of work items) of the k-th item of CTA c among G, or n when CTA c has
// fewer than k + 1 items.  With a schedule -- offsets sched[0..G], then the
// items of CTA c at sched[G + 1 + sched[c]] .. sched[G + 1 + sched[c + 1] - 1],
// packed on the host -- its entries.  Otherwise rounds of G items dealt
// c = 0..G-1 in even rounds and G-1..0 in odd rounds, so that long and short
// items mix: over all n indices, or, for a packed (varlen) batch, over the
// list compact[1 .. compact[0]] of the items that are not empty (a short
// sequence has no items for the higher blocks; dealt with their holes, they
// left some CTAs with far more work than others).
__device__ __forceinline__ int dealt_item(const int* sched, const int* compact, int k, int c,
                                          int G, int n) {
  if (sched) {
    const int b = __ldg(sched + c), e = __ldg(sched + c + 1);
    return b + k < e ? __ldg(sched + G + 1 + b + k) : n;
  }
  const int m = k * G + ((k & 1) ? (G - 1 - c) : c);
  if (compact) return m < __ldg(compact) ? __ldg(compact + 1 + m) : n;
  return m < n ? m : n;
}

// Parameters of the projection GEMM (ne_proj.cu), shared by the launches in
// the API file.
namespace gemm {
enum Epilogue { kQkvRope = 0, kResidual = 1, kMtpCe = 2, kScale = 3, kReduceF32 = 4 };
struct Params {
  int M = 0, N = 0, K = 0;
  int n_tiles_m = 0, n_tiles_n = 0;
  int tile_n = 256;               // output tile width (256; 192 for kResidual / kScale)
  int k_splits = 1;               // K ranges per output tile (more than 1: kReduceF32 only)
  int chunks_per_split = 1 << 20;  // 64-wide K chunks per range
  int C = 0;  // kQkvRope: width of each of q, k, v (N = 3C)
  int T = 1;  // kQkvRope: tokens per sequence (position = row mod T)
  RopeTable rope{nullptr, nullptr, 0};
  // Multi-token prediction head
  const int* targets = nullptr;  // [M, heads] (kMtpCe): token id, or -1 for no target
  int heads = 1;                 // kMtpCe: heads of 256 logits (N = 256 * heads)
  float* row_loss = nullptr;     // [M, heads] (kMtpCe)
  float* acc = nullptr;          // [2]: sum of the row losses, count of targets (kMtpCe adds)
  float* loss = nullptr;         // [1]: acc[0] / acc[1], written by kScale
  int* status = nullptr;
};
}  // namespace gemm

// Index of LSE / delta element (head h, sequence s starting at row `start`,
// position t within the sequence).
__device__ __forceinline__ long long lse_index(const Problem& pb, int h, int s, int start, int t) {
  if (pb.lse_fixed) return (static_cast<long long>(s) * pb.H + h) * pb.max_len + t;
  return static_cast<long long>(h) * pb.n_tot + start + t;
}

}  // namespace ne
