// ne_attn_noalloc.cu -- ne_attn_bwd_noalloc: the backward for callers that can
// allocate no device memory (see include/ne_attn.h).  Everything the backward
// needs beyond its inputs and outputs -- the RoPE cos/sin table, the fp32 dQ'
// accumulator, the D_m row terms and the rotated copies q', k' -- lives in one
// file-scope device array owned by the library.  It launches the same kernels as ne_attn_bwd.
#include <cmath>
#include <cstring>
#include <mutex>

#include "ne_attn.h"
#include "ne_common.cuh"

namespace ne {
cudaError_t launch_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmDO, const CUtensorMap& tmDQ, const CUtensorMap& tmDV,
                       const CUtensorMap& tmDK, const BwdParams& p, int n_tiles,
                       cudaStream_t stream, cudaEvent_t ev_pre, cudaEvent_t ev_main);
ne_status internal_prepare(int** status_word);
ne_status internal_encode_rows(CUtensorMap* map, const void* base, int n_rows, int H);
ne_status internal_encode_rows_f32(CUtensorMap* map, void* base, int n_rows, int H);
}  // namespace ne

namespace {

// Layout of the scratch: [RoPE table: positions x 32 (cos, sin)] [dQ' fp32
// accumulator: rows x 64] [D_m: rows] [q' bf16: rows x 64] [k' bf16: rows x
// 64], each part 256-byte aligned.
constexpr size_t kScratchBytes = NE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxPositions = NE_NOALLOC_MAX_POSITIONS;
constexpr long long kMaxRows = NE_NOALLOC_MAX_ROWS;
constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
constexpr size_t kTableBytes = align256(static_cast<size_t>(kMaxPositions) * 32 * sizeof(float2));
static_assert(kTableBytes + align256(kMaxRows * 64 * sizeof(float)) +
                      align256(kMaxRows * sizeof(float)) + 2 * align256(kMaxRows * 64 * 2) <=
                  kScratchBytes,
              "scratch too small for the stated limits");

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; the device address is obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct NoAllocDevice {
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  float table_base = 0.f;            // rope_base the table currently holds (0: none)
};
std::mutex g_noalloc_mutex;
NoAllocDevice g_noalloc_dev[kMaxDevices];

// The RoPE table for `base`, built on the host in double with the same rule as
// the library's cached tables (cs[p * 32 + i] = fp32 cos / sin of p * theta_i,
// theta_i = base^(-(2i)/64)), and copied into the scratch with one copy
// enqueued on `stream`.  Being stream-ordered, the copy starts only after the
// kernels of earlier calls on this stream, which read the old table, have
// finished, and the kernels this call launches next see the new table.  The
// host image is a pageable array: an asynchronous copy from pageable memory
// has taken its bytes by the time it returns, so the image may be rebuilt by
// the next call at once.
ne_status upload_table(unsigned char* dst, float base, cudaStream_t stream) {
  static float2 image[static_cast<size_t>(kMaxPositions) * 32];
  double theta[32];
  for (int i = 0; i < 32; ++i) theta[i] = std::pow(static_cast<double>(base), -(2.0 * i) / 64.0);
  for (int p = 0; p < kMaxPositions; ++p)
    for (int i = 0; i < 32; ++i) {
      const double a = static_cast<double>(p) * theta[i];
      image[static_cast<size_t>(p) * 32 + i] =
          make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
    }
  if (cudaMemcpyAsync(dst, image, sizeof(image), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return NE_ERR_CUDA;
  return NE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ne_status ne_attn_bwd_noalloc(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                                         const ne_bf16* out, const ne_bf16* dout,
                                         const float* lse, int B, int H, int T, int D,
                                         float rope_base, float scale, ne_bf16* dq, ne_bf16* dk,
                                         ne_bf16* dv, void* stream) {
  // ---- host-side checks, before the device is touched ----------------------
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return NE_ERR_INVALID_ARG;
  if (D != 64) return NE_ERR_UNSUPPORTED;
  if (B <= 0 || H <= 0 || T <= 0) return NE_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale <= 0.f || !std::isfinite(rope_base) || rope_base <= 0.f)
    return NE_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * T * H;
  if (T > kMaxPositions || rows > kMaxRows) return NE_ERR_TOO_LARGE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return NE_ERR_MISALIGNED;

  int* status = nullptr;
  ne_status rc = ne::internal_prepare(&status);
  if (rc != NE_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NE_ERR_CUDA;

  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoAllocDevice& nd = g_noalloc_dev[dev];
  if (!nd.scratch) {  // once per device, with that device current
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NE_ERR_CUDA;
    nd.scratch = static_cast<unsigned char*>(ptr);
  }
  if (nd.table_base != rope_base) {
    // A copy captured into a graph would read the host image at replay time,
    // when later calls may have rebuilt it for another base: refused.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capture) != cudaSuccess)
      return NE_ERR_CUDA;
    if (capture != cudaStreamCaptureStatusNone) return NE_ERR_UNSUPPORTED;
    nd.table_base = 0.f;
    if ((rc = upload_table(nd.scratch, rope_base, static_cast<cudaStream_t>(stream))) != NE_OK)
      return rc;
    nd.table_base = rope_base;
  }

  const int n_tot = B * T;
  const int n_tiles = (T + 127) / 128;
  ne::BwdParams p;
  p.pb.cu_seqlens = nullptr;
  p.pb.nseq = B;
  p.pb.max_len = T;
  p.pb.H = H;
  p.pb.n_tot = n_tot;
  p.pb.lse_fixed = 1;
  p.out = reinterpret_cast<const __nv_bfloat16*>(out);
  p.dout = reinterpret_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.dq = reinterpret_cast<__nv_bfloat16*>(dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(dv);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status;
  p.rope.cs = reinterpret_cast<const float2*>(nd.scratch);
  p.rope.csw = nullptr;  // the backward reads the row layout only
  p.rope.capacity = kMaxPositions;
  p.rotate_in = 1;
  p.rotate_out = 1;
  // The preprocess kernel of every call zeroes the dQ' accumulator and
  // overwrites D_m, q' and k', so nothing left by an earlier call is read.
  const size_t acc_bytes = align256(static_cast<size_t>(rows) * 64 * sizeof(float));
  const size_t del_bytes = align256(static_cast<size_t>(rows) * sizeof(float));
  const size_t rot_bytes = align256(static_cast<size_t>(rows) * 64 * 2);
  unsigned char* w = nd.scratch + kTableBytes;
  p.dq_acc = reinterpret_cast<float*>(w);
  p.delta = reinterpret_cast<float*>(w + acc_bytes);
  p.qr = reinterpret_cast<__nv_bfloat16*>(w + acc_bytes + del_bytes);
  p.kr = reinterpret_cast<__nv_bfloat16*>(w + acc_bytes + del_bytes + rot_bytes);
  p.q = reinterpret_cast<const __nv_bfloat16*>(q);
  p.k = reinterpret_cast<const __nv_bfloat16*>(k);

  CUtensorMap tq, tk, tv, tdo, tdq;
  if ((rc = ne::internal_encode_rows(&tq, p.qr, n_tot, H)) != NE_OK) return rc;
  if ((rc = ne::internal_encode_rows(&tk, p.kr, n_tot, H)) != NE_OK) return rc;
  if ((rc = ne::internal_encode_rows(&tv, v, n_tot, H)) != NE_OK) return rc;
  if ((rc = ne::internal_encode_rows(&tdo, dout, n_tot, H)) != NE_OK) return rc;
  if ((rc = ne::internal_encode_rows_f32(&tdq, p.dq_acc, n_tot, H)) != NE_OK) return rc;
  CUtensorMap tdv, tdk;
  if ((rc = ne::internal_encode_rows(&tdv, dv, n_tot, H)) != NE_OK) return rc;
  if ((rc = ne::internal_encode_rows(&tdk, dk, n_tot, H)) != NE_OK) return rc;
  const cudaError_t e = ne::launch_bwd(tq, tk, tv, tdo, tdq, tdv, tdk, p, n_tiles,
                                       static_cast<cudaStream_t>(stream), nullptr, nullptr);
  if (e == cudaSuccess) return NE_OK;
  return e == cudaErrorMemoryAllocation ? NE_ERR_OOM : NE_ERR_CUDA;
}
