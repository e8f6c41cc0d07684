// ne_attn_api.cu -- the C ABI (include/ne_attn.h, include/ne_attn_debug.h):
// host-side argument checks, TMA tensor-map encoding, the per-device RoPE
// cos/sin table cache, the device status word, backward workspace handling,
// and the launches.  No arithmetic of the method runs here except building the
// RoPE table (on the host, in double).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "ne_attn.h"
#include "ne_attn_debug.h"
#include "ne_common.cuh"

namespace ne {
cudaError_t launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmO, const FwdParams& p, int n_qtiles,
                       cudaStream_t stream);
cudaError_t launch_rope_rows(const __nv_bfloat16* x0, __nv_bfloat16* xr0,
                             const __nv_bfloat16* x1, __nv_bfloat16* xr1, const Problem& pb,
                             const RopeTable& rope, cudaStream_t stream);
cudaError_t launch_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmDO, const CUtensorMap& tmDQ, const CUtensorMap& tmDV,
                       const CUtensorMap& tmDK, const BwdParams& p, int n_tiles,
                       cudaStream_t stream, cudaEvent_t ev_pre, cudaEvent_t ev_main);
cudaError_t launch_debug_tile(const CUtensorMap& tm, int h, int row0, int rotate, int pos0,
                              RopeTable rope, void* dst_raw, __nv_bfloat16* dst_rows,
                              int* status, cudaStream_t stream);
cudaError_t launch_debug_umma(int form, const __nv_bfloat16* a, const __nv_bfloat16* b, float* d,
                              int* status, cudaStream_t stream);
cudaError_t launch_debug_pipeline(const CUtensorMap& tm, int n_items, int drop_item,
                                  long long limit, float* d, int* status, cudaStream_t stream);
std::vector<int> unit_steps(int nseq, int H, int T);
cudaError_t launch_compact_items(const Problem& pb, int kind, int n_blocks, int n_buckets,
                                 int* out, cudaStream_t stream);
std::vector<int> pack_schedule(const std::vector<int>& w, int G, double c_lo, double c_hi);
size_t decode_part_bytes(int B, int H, int Tmax);
cudaError_t launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmT,
                          const __nv_bfloat16* q, const int* pos, int B, int H, int Tmax,
                          const RopeTable& rope, float scale_log2, float* part,
                          __nv_bfloat16* out, float* lse, int* status, cudaStream_t stream,
                          bool rot);
constexpr unsigned kDecodeBoxRows = 32;  // keys per pipeline stage of the decode kernel
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* xn,
                           float* rstd, int M, int C, float eps, cudaStream_t stream);
int gemm_tile_n(int epi, long long M, int N, int G);
cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const CUtensorMap& tmO0, const CUtensorMap& tmO1, const CUtensorMap& tmO2,
                        const gemm::Params& p, cudaStream_t stream);
}  // namespace ne

namespace {

using ne::RopeTable;

__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;

struct RopeEntry {
  float base = 0.f;
  int capacity = 0;
  float2* dev = nullptr;
};

// A temporary the forward keeps per stream (the rotated keys k'): allocated
// on that stream the first time, grown (stream-ordered) when a larger problem
// comes, reused by every later call on the stream, whose kernels it orders.
struct StreamScratch {
  cudaStream_t stream = nullptr;
  void* ptr = nullptr;
  size_t bytes = 0;
};

// A work schedule of the persistent backward for one fixed-length shape
// (ne_sched.cu); dev == nullptr where the snake order is kept.
struct SchedEntry {
  int nseq = 0, H = 0, T = 0, G = 0;
  int* dev = nullptr;
};

struct DeviceState {
  bool ready = false;
  int* status = nullptr;  // device address of g_device_status on this device
  bool supported = false;
  int sm_count = 0;
  std::vector<RopeEntry> tables;
  std::vector<float2*> retired;  // replaced tables, freed by ne_attn_release
  std::vector<StreamScratch> scratch;
  std::vector<SchedEntry> scheds;
};

// The forward's per-stream temporary of at least `bytes` (caller holds g_mutex).
ne_status stream_scratch(DeviceState& st, cudaStream_t stream, size_t bytes, void** out) {
  for (auto& e : st.scratch)
    if (e.stream == stream) {
      if (e.bytes < bytes) {
        // Enqueued after every earlier use of the old buffer on this stream.
        if (cudaFreeAsync(e.ptr, stream) != cudaSuccess) return NE_ERR_CUDA;
        e.ptr = nullptr;
        e.bytes = 0;
        cudaError_t r = cudaMallocAsync(&e.ptr, bytes, stream);
        if (r != cudaSuccess) return r == cudaErrorMemoryAllocation ? NE_ERR_OOM : NE_ERR_CUDA;
        e.bytes = bytes;
      }
      *out = e.ptr;
      return NE_OK;
    }
  StreamScratch e;
  e.stream = stream;
  cudaError_t r = cudaMallocAsync(&e.ptr, bytes, stream);
  if (r != cudaSuccess) return r == cudaErrorMemoryAllocation ? NE_ERR_OOM : NE_ERR_CUDA;
  e.bytes = bytes;
  st.scratch.push_back(e);
  *out = e.ptr;
  return NE_OK;
}

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
int g_last_code = 0;
cudaEvent_t g_ev_pre = nullptr, g_ev_main = nullptr, g_ev_rot = nullptr;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

ne_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NE_OK;
  if (e == cudaErrorMemoryAllocation) return NE_ERR_OOM;
  return NE_ERR_CUDA;
}

// Per-device set-up (caller holds g_mutex).
ne_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NE_ERR_UNSUPPORTED;
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NE_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return NE_ERR_CUDA;
    st.status = static_cast<int*>(p);
    st.ready = true;
  }
  if (!st.supported) return NE_ERR_UNSUPPORTED;
  *out = &st;
  return NE_OK;
}

ne_status get_encoder() {
  if (g_encode) return NE_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return NE_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return NE_OK;
}

RopeTable table_view(float2* dev, int cap) {
  return RopeTable{dev, reinterpret_cast<const float4*>(dev + static_cast<size_t>(cap) * 32), cap};
}

// RoPE table for (base, D = 64) covering at least `positions` positions:
// cs[p * 32 + i] = ((float)cos(p * theta_i), (float)sin(p * theta_i)),
// theta_i = base^(-(2i)/64), all in double before the final fp32 rounding;
// followed by the same values in the warp-interleaved layout of RopeTable::csw.
ne_status rope_table(DeviceState& st, float base, int positions, cudaStream_t stream,
                     RopeTable* out) {
  for (auto& e : st.tables)
    if (e.base == base && e.capacity >= positions) {
      *out = table_view(e.dev, e.capacity);
      return NE_OK;
    }
  // A new table is built with a synchronous allocation and copy, which a
  // stream capture does not allow: the first call for a base (or for more
  // positions) must run outside the capture.
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return NE_ERR_CUDA;
  if (capture != cudaStreamCaptureStatusNone) return NE_ERR_UNSUPPORTED;
  int cap = 4096;
  while (cap < positions) cap *= 2;
  std::vector<float2> host(static_cast<size_t>(cap) * 64);
  float2* inter = host.data() + static_cast<size_t>(cap) * 32;
  for (int i = 0; i < 32; ++i) {
    const double theta = std::pow(static_cast<double>(base), -(2.0 * i) / 64.0);
    for (int pos = 0; pos < cap; ++pos) {
      const double a = static_cast<double>(pos) * theta;
      const float2 v =
          make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
      host[static_cast<size_t>(pos) * 32 + i] = v;
      // float4 (i / 2) of position pos = 32 g + l sits at ((16 g + i / 2) * 32 + l).
      const size_t q4 = (static_cast<size_t>(pos >> 5) * 16 + (i >> 1)) * 32 + (pos & 31);
      inter[q4 * 2 + (i & 1)] = v;
    }
  }
  float2* dev = nullptr;
  cudaError_t e = cudaMalloc(&dev, host.size() * sizeof(float2));
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemcpy(dev, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(dev);
    return cuda_status(e);
  }
  for (auto& t : st.tables)
    if (t.base == base) {
      // Kernels already enqueued may still read the old table: retire it.
      st.retired.push_back(t.dev);
      t.dev = dev;
      t.capacity = cap;
      *out = table_view(dev, cap);
      return NE_OK;
    }
  st.tables.push_back(RopeEntry{base, cap, dev});
  *out = table_view(dev, cap);
  return NE_OK;
}

// Per-unit overhead range of the persistent backward, in query-tile steps:
// fits of unit duration = overhead + steps x step time to globaltimer stamps
// of every CTA on GB300 give 1.2-1.8 steps (the unit's K', V loads and its
// dV/dK epilogue) at the GPT-2-small, 4096 and 16384-byte shapes.
constexpr double kBwdOverhead[2] = {1.0, 2.0};
constexpr size_t kMaxSchedules = 256;

// The work schedule of the persistent backward (its units over n_tiles x nseq
// x H) for a fixed-length batch of length T: packed on the host on first use
// of the shape and kept on the device.  *sched = nullptr keeps the kernel's
// snake order: when it is as good, for a packed (varlen) batch, or when a
// table cannot be made now (the stream is being captured, or the cache is
// full).
ne_status work_schedule(DeviceState& st, bool fixed, int nseq, int H, int T, cudaStream_t stream,
                        const int** sched, int* G) {
  *sched = nullptr;
  *G = 0;
  if (!fixed) return NE_OK;
  const long long n = static_cast<long long>((T + 127) / 128) * nseq * H;
  *G = static_cast<int>(n < st.sm_count ? n : st.sm_count);
  for (const auto& e : st.scheds)
    if (e.nseq == nseq && e.H == H && e.T == T && e.G == *G) {
      *sched = e.dev;
      return NE_OK;
    }
  if (st.scheds.size() >= kMaxSchedules) return NE_OK;
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) return NE_ERR_CUDA;
  if (capture != cudaStreamCaptureStatusNone) return NE_OK;
  const std::vector<int> tab =
      ne::pack_schedule(ne::unit_steps(nseq, H, T), *G, kBwdOverhead[0], kBwdOverhead[1]);
  SchedEntry e;
  e.nseq = nseq;
  e.H = H;
  e.T = T;
  e.G = *G;
  if (!tab.empty()) {
    cudaError_t r = cudaMalloc(&e.dev, tab.size() * sizeof(int));
    if (r == cudaSuccess)
      r = cudaMemcpy(e.dev, tab.data(), tab.size() * sizeof(int), cudaMemcpyHostToDevice);
    if (r != cudaSuccess) {
      if (e.dev) cudaFree(e.dev);
      return cuda_status(r);
    }
  }
  st.scheds.push_back(e);
  *sched = e.dev;
  return NE_OK;
}

// 3-d tensor map over [n_rows, H, 64] bf16, box 64 x 1 x 128, 128-byte swizzle.
ne_status encode_rows(CUtensorMap* map, const void* base, int n_rows, int H,
                      unsigned box_rows = 128) {
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n_rows)};
  cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(H) * 64 * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 3-d tensor map over the fp32 dQ' accumulator [n_rows, H, 64], box 32 x 1 x 128
// (128-byte rows), 128-byte swizzle: the target of the backward's bulk reduce-adds.
ne_status encode_rows_f32(CUtensorMap* map, void* base, int n_rows, int H) {
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(n_rows)};
  cuuint64_t strides[2] = {64 * 4, static_cast<cuuint64_t>(H) * 64 * 4};
  cuuint32_t box[3] = {32, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 2-d tensor map over the RoPE table's row layout: `positions` rows of 64
// fp32 (32 (cos, sin) pairs), box 32 x `box_rows` (one 128-byte half row per
// box row), 128-byte swizzle.
ne_status encode_table(CUtensorMap* map, const float2* cs, int positions, unsigned box_rows) {
  cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(positions)};
  cuuint64_t strides[1] = {64 * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                        const_cast<void*>(static_cast<const void*>(cs)), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 2-d tensor map over a row-major [rows, cols] bf16 matrix, box 64 x box_rows,
// 128-byte swizzle (the operand and output tiles of the projection GEMM).
ne_status encode_mat(CUtensorMap* map, const void* base, long long rows, int cols,
                     unsigned box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// fp32 [rows, cols] matrix, boxes of 32 columns (128 bytes) x box_rows.
ne_status encode_mat_f32(CUtensorMap* map, void* base, long long rows, int cols,
                         unsigned box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Shape {
  const int* cu = nullptr;
  int nseq = 0, n_tot = 0, max_len = 0, H = 0, D = 0;
  bool fixed = true;
};

ne_status check_shape(const Shape& s) {
  if (s.D != 64) return NE_ERR_UNSUPPORTED;
  if (s.H <= 0 || s.nseq <= 0 || s.max_len <= 0 || s.n_tot <= 0) return NE_ERR_INVALID_ARG;
  if (!s.fixed && !s.cu) return NE_ERR_INVALID_ARG;
  const long long rows = s.fixed ? static_cast<long long>(s.nseq) * s.max_len : s.n_tot;
  if (rows > (1LL << 31) - 1 - 256) return NE_ERR_INVALID_ARG;
  if (static_cast<long long>(s.nseq) * s.H > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  if ((s.max_len + 127) / 128 > 65535) return NE_ERR_INVALID_ARG;
  // Every (row, head) pair index fits in 32 bits (each tensor then stays under
  // 256 GB, more than the device holds).
  if (static_cast<long long>(rows) * s.H > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return NE_OK;
}

ne::Problem make_problem(const Shape& s) {
  ne::Problem pb;
  pb.cu_seqlens = s.fixed ? nullptr : s.cu;
  pb.nseq = s.nseq;
  pb.max_len = s.max_len;
  pb.H = s.H;
  pb.n_tot = s.n_tot;
  pb.lse_fixed = s.fixed ? 1 : 0;
  return pb;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Packed (varlen) batches: the persistent kernels deal the non-empty items of
// their work lists, longest first, as sorted on the device by a one-CTA
// kernel (ne_sched.cu) into a per-stream temporary, up to this many items
// (beyond, that single CTA would take longer than the imbalance it removes
// may save; the kernels then deal the whole list).
constexpr long long kMaxCompactItems = 1 << 16;
constexpr int kMaxBuckets = 8192;  // its counting sort's buckets (shared memory, 32 KB)

// Sequence length from which the forward rotates the keys once per call in a
// pass of its own instead of in every item that uses a key tile (measured on
// GB300: below it the extra pass costs more than the kernel saves).
constexpr int kPreRotateLen = 2048;

// How the operands are rotated.  kRotate: q, k as given, rotated inside;
// kPreRotated: q, k are q' = R(m) q, k' = R(n) k already (rope_base unused);
// kTrain: q, k as given, rotated by one pass into the caller's qr, kr, which
// the attention kernel then reads (and the backward later reuses).
enum class Rot { kRotate, kPreRotated, kTrain };

ne_status run_fwd(const Shape& s, const void* q, const void* k, const void* v, float rope_base,
                  float scale, void* out, int out_f32, float* lse, void* stream,
                  Rot mode = Rot::kRotate, void* qr_out = nullptr, void* kr_out = nullptr) {
  const bool pre_rotated = mode == Rot::kPreRotated;
  if (!q || !k || !v || !out || !lse) return NE_ERR_INVALID_ARG;
  if (mode == Rot::kTrain && (!qr_out || !kr_out)) return NE_ERR_INVALID_ARG;
  if (mode == Rot::kTrain && (!aligned16(qr_out) || !aligned16(kr_out))) return NE_ERR_MISALIGNED;
  ne_status rc = check_shape(s);
  if (rc != NE_OK) return rc;
  if (!std::isfinite(scale) || scale <= 0.f ||
      (!pre_rotated && (!std::isfinite(rope_base) || rope_base <= 0.f)))
    return NE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned4(lse))
    return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  const int n_qtiles = (s.max_len + 127) / 128;
  ne::FwdParams p;
  p.pb = make_problem(s);
  p.out = out;
  p.out_f32 = out_f32;
  p.lse = lse;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = st->status;
  p.rope = RopeTable{nullptr, nullptr, 0};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (!pre_rotated && (rc = rope_table(*st, rope_base, n_qtiles * 128, cs, &p.rope)) != NE_OK)
    return rc;
  // Keys: for short sequences each item rotates the key tiles it uses in
  // shared memory; from kPreRotateLen positions on, the rotated keys
  // k' = R(n) k are written once per call by a small pass into the library's
  // temporary for this stream, or, while the stream is being captured into a
  // graph, into a stream-ordered allocation of the call's own (a graph must
  // not bake in a buffer that later calls outside it would also use).
  p.rotate_k = (mode == Rot::kRotate && s.max_len < kPreRotateLen) ? 1 : 0;
  p.rotate_q = mode == Rot::kRotate ? 1 : 0;
  CUtensorMap tq, tk, tv, to;
  const void* queries = mode == Rot::kTrain ? qr_out : q;
  const void* keys = mode == Rot::kTrain ? kr_out : k;
  // Temporaries: the rotated keys (long sequences) and, for a packed batch,
  // the compacted item list.
  const int nblk = (n_qtiles + 1) / 2;
  const long long n_items = static_cast<long long>(nblk) * s.nseq * s.H;
  const bool compact = !s.fixed && n_items <= kMaxCompactItems && 2 * nblk + 1 <= kMaxBuckets;
  const size_t kr_bytes =
      (mode == Rot::kRotate && !p.rotate_k) ? static_cast<size_t>(s.n_tot) * s.H * 64 * 2 : 0;
  const size_t tmp_bytes =
      align256(kr_bytes) + (compact ? static_cast<size_t>(n_items + 1) * sizeof(int) : 0);
  bool own = false;
  void* tmp = nullptr;
  void* kr = nullptr;
  int* list = nullptr;
  cudaError_t e = cudaSuccess;
  if (tmp_bytes) {
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &capture) != cudaSuccess) return NE_ERR_CUDA;
    own = capture != cudaStreamCaptureStatusNone;
    if (own) {
      if ((e = cudaMallocAsync(&tmp, tmp_bytes, cs)) != cudaSuccess) return cuda_status(e);
    } else if ((rc = stream_scratch(*st, cs, tmp_bytes, &tmp)) != NE_OK) {
      return rc;
    }
    if (kr_bytes) {
      kr = tmp;
      keys = kr;
    }
    if (compact) list = reinterpret_cast<int*>(static_cast<char*>(tmp) + align256(kr_bytes));
  }
  rc = encode_rows(&tq, queries, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows(&tk, keys, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows(&tv, v, s.n_tot, s.H);
  // O tile stores (bf16 output only; the fp32 output is written per row).
  if (rc == NE_OK) rc = encode_rows(&to, out_f32 ? q : out, s.n_tot, s.H);
  if (rc == NE_OK) {
    if (mode == Rot::kRotate && !p.rotate_k)
      e = ne::launch_rope_rows(static_cast<const __nv_bfloat16*>(k),
                               static_cast<__nv_bfloat16*>(kr), nullptr, nullptr, p.pb, p.rope,
                               cs);
    else if (mode == Rot::kTrain)
      e = ne::launch_rope_rows(static_cast<const __nv_bfloat16*>(q),
                               static_cast<__nv_bfloat16*>(qr_out),
                               static_cast<const __nv_bfloat16*>(k),
                               static_cast<__nv_bfloat16*>(kr_out), p.pb, p.rope, cs);
    const bool pass = (mode == Rot::kRotate && !p.rotate_k) || mode == Rot::kTrain;
    if (e == cudaSuccess && g_ev_rot && pass) e = cudaEventRecord(g_ev_rot, cs);
    if (e == cudaSuccess && compact) {
      e = ne::launch_compact_items(p.pb, 0, nblk, 2 * nblk + 1, list, cs);
      p.compact = list;
    }
    if (e == cudaSuccess) e = ne::launch_fwd(tq, tk, tv, to, p, n_qtiles, cs);
  }
  if (own) {
    const cudaError_t e2 = cudaFreeAsync(tmp, cs);
    if (e == cudaSuccess) e = e2;
  }
  if (rc != NE_OK) return rc;
  return cuda_status(e);
}

// kRotate: q, k as given; kPreRotated: q, k are q', k' and the gradients
// returned are w.r.t. them; kTrain: q, k are q', k' (from the training
// forward) and the gradients returned are w.r.t. the un-rotated q, k.
ne_status run_bwd(const Shape& s, const void* q, const void* k, const void* v, const void* out,
                  const void* dout, const float* lse, float rope_base, float scale, void* dq,
                  void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream,
                  Rot mode = Rot::kRotate) {
  const bool pre_rotated = mode == Rot::kPreRotated;
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return NE_ERR_INVALID_ARG;
  ne_status rc = check_shape(s);
  if (rc != NE_OK) return rc;
  if (!std::isfinite(scale) || scale <= 0.f ||
      (!pre_rotated && (!std::isfinite(rope_base) || rope_base <= 0.f)))
    return NE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned4(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return NE_ERR_MISALIGNED;
  const size_t need = ne_attn_bwd_workspace_bytes(s.n_tot, s.H, s.D);
  if (workspace && workspace_bytes < need) return NE_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  if ((rc = device_state(&st)) != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int n_tiles = (s.max_len + 127) / 128;
  ne::BwdParams p;
  p.pb = make_problem(s);
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = st->status;
  p.rotate_in = mode == Rot::kRotate ? 1 : 0;
  p.rotate_out = pre_rotated ? 0 : 1;
  p.rope = RopeTable{nullptr, nullptr, 0};
  if (!pre_rotated && (rc = rope_table(*st, rope_base, n_tiles * 128, cs, &p.rope)) != NE_OK)
    return rc;
  if ((rc = work_schedule(*st, s.fixed, s.nseq, s.H, s.max_len, cs, &p.sched, &p.sched_ctas)) !=
      NE_OK)
    return rc;
  CUtensorMap tq, tk, tv, tdo;
  if ((rc = encode_rows(&tv, v, s.n_tot, s.H)) != NE_OK) return rc;
  if ((rc = encode_rows(&tdo, dout, s.n_tot, s.H)) != NE_OK) return rc;
  void* ws = workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, cs);
    if (e != cudaSuccess) return cuda_status(e);
    owned = true;
  }
  // Workspace: [dQ' fp32][D fp32][q' bf16][k' bf16], each part 256-byte aligned.
  const size_t acc_bytes = align256(static_cast<size_t>(s.n_tot) * s.H * 64 * sizeof(float));
  const size_t del_bytes = align256(static_cast<size_t>(s.n_tot) * s.H * sizeof(float));
  const size_t rot_bytes = align256(static_cast<size_t>(s.n_tot) * s.H * 64 * 2);
  char* wsb = static_cast<char*>(ws);
  p.dq_acc = reinterpret_cast<float*>(wsb);
  p.delta = reinterpret_cast<float*>(wsb + acc_bytes);
  p.qr = reinterpret_cast<__nv_bfloat16*>(wsb + acc_bytes + del_bytes);
  p.kr = reinterpret_cast<__nv_bfloat16*>(wsb + acc_bytes + del_bytes + rot_bytes);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  if (!p.rotate_in) {  // the main kernel reads q', k' where the caller keeps them
    p.qr = const_cast<__nv_bfloat16*>(p.q);
    p.kr = const_cast<__nv_bfloat16*>(p.k);
  }
  // Packed batch: the compacted unit list in the library's temporary for this
  // stream (a stream-ordered allocation of the call's own during capture).
  const long long n_units = static_cast<long long>(n_tiles) * s.nseq * s.H;
  const bool compact = !s.fixed && n_units <= kMaxCompactItems && n_tiles + 1 <= kMaxBuckets;
  int* list = nullptr;
  bool own_list = false;
  if (compact) {
    const size_t list_bytes = static_cast<size_t>(n_units + 1) * sizeof(int);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(cs, &capture) != cudaSuccess) rc = NE_ERR_CUDA;
    own_list = capture != cudaStreamCaptureStatusNone;
    void* lp = nullptr;
    if (rc == NE_OK) {
      if (own_list) {
        const cudaError_t e = cudaMallocAsync(&lp, list_bytes, cs);
        if (e != cudaSuccess) rc = cuda_status(e);
      } else {
        rc = stream_scratch(*st, cs, list_bytes, &lp);
      }
    }
    list = static_cast<int*>(lp);
    if (rc != NE_OK) own_list = false;
  }
  CUtensorMap tdq, tdv, tdk;
  if (rc == NE_OK) rc = encode_rows(&tq, p.qr, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows(&tk, p.kr, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows_f32(&tdq, p.dq_acc, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows(&tdv, dv, s.n_tot, s.H);
  if (rc == NE_OK) rc = encode_rows(&tdk, dk, s.n_tot, s.H);
  cudaError_t e = cudaSuccess;
  if (rc == NE_OK && compact) {
    e = ne::launch_compact_items(p.pb, 1, n_tiles, n_tiles + 1, list, cs);
    p.compact = list;
  }
  if (rc == NE_OK && e == cudaSuccess)
    e = ne::launch_bwd(tq, tk, tv, tdo, tdq, tdv, tdk, p, n_tiles, cs, g_ev_pre, g_ev_main);
  else if (rc != NE_OK)
    e = cudaErrorInvalidValue;
  if (own_list) {
    const cudaError_t e2 = cudaFreeAsync(list, cs);
    if (e == cudaSuccess) e = e2;
  }
  if (owned) {
    cudaError_t e2 = cudaFreeAsync(ws, cs);
    if (e == cudaSuccess) e = e2;
  }
  if (rc != NE_OK) return rc;
  return cuda_status(e);
}

}  // namespace

namespace ne {
// Helpers for the allocation-free backward entry point (ne_attn_noalloc.cu):
// per-device set-up, the device status word, and the tensor-map encoders.
ne_status internal_prepare(int** status_word) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  *status_word = st->status;
  return NE_OK;
}
ne_status internal_encode_rows(CUtensorMap* map, const void* base, int n_rows, int H) {
  return encode_rows(map, base, n_rows, H);
}
ne_status internal_encode_rows_f32(CUtensorMap* map, void* base, int n_rows, int H) {
  return encode_rows_f32(map, base, n_rows, H);
}
}  // namespace ne

extern "C" {

const char* ne_status_string(ne_status s) {
  switch (s) {
    case NE_OK: return "NE_OK";
    case NE_ERR_INVALID_ARG: return "NE_ERR_INVALID_ARG";
    case NE_ERR_UNSUPPORTED: return "NE_ERR_UNSUPPORTED";
    case NE_ERR_MISALIGNED: return "NE_ERR_MISALIGNED";
    case NE_ERR_CUDA: return "NE_ERR_CUDA";
    case NE_ERR_TIMEOUT: return "NE_ERR_TIMEOUT";
    case NE_ERR_OOM: return "NE_ERR_OOM";
    case NE_ERR_BAD_SEQLEN: return "NE_ERR_BAD_SEQLEN";
    case NE_ERR_TOO_LARGE: return "NE_ERR_TOO_LARGE";
    default: return "NE_ERR_UNKNOWN";
  }
}

size_t ne_attn_bwd_workspace_bytes(int n_tot, int H, int D) {
  if (n_tot <= 0 || H <= 0 || D != 64) return 0;
  return align256(static_cast<size_t>(n_tot) * H * 64 * sizeof(float)) +
         align256(static_cast<size_t>(n_tot) * H * sizeof(float)) +
         2 * align256(static_cast<size_t>(n_tot) * H * 64 * 2);
}

ne_status ne_attn_fwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H, int T,
                      int D, float rope_base, float scale, ne_bf16* out, float* lse,
                      void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_fwd(s, q, k, v, rope_base, scale, out, 0, lse, stream);
}

ne_status ne_attn_fwd_f32out(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H,
                             int T, int D, float rope_base, float scale, float* out, float* lse,
                             void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_fwd(s, q, k, v, rope_base, scale, out, 1, lse, stream);
}

ne_status ne_attn_varlen_fwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                             const int* cu_seqlens, int nseq, int n_tot, int max_seqlen, int H,
                             int D, float rope_base, float scale, ne_bf16* out, float* lse,
                             void* stream) {
  Shape s;
  s.cu = cu_seqlens;
  s.fixed = false;
  s.nseq = nseq;
  s.n_tot = n_tot;
  s.max_len = max_seqlen;
  s.H = H;
  s.D = D;
  return run_fwd(s, q, k, v, rope_base, scale, out, 0, lse, stream);
}

ne_status ne_attn_varlen_fwd_f32out(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                                    const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                    int H, int D, float rope_base, float scale, float* out,
                                    float* lse, void* stream) {
  Shape s;
  s.cu = cu_seqlens;
  s.fixed = false;
  s.nseq = nseq;
  s.n_tot = n_tot;
  s.max_len = max_seqlen;
  s.H = H;
  s.D = D;
  return run_fwd(s, q, k, v, rope_base, scale, out, 1, lse, stream);
}

ne_status ne_attn_bwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, const ne_bf16* out,
                      const ne_bf16* dout, const float* lse, int B, int H, int T, int D,
                      float rope_base, float scale, ne_bf16* dq, ne_bf16* dk, ne_bf16* dv,
                      void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_bwd(s, q, k, v, out, dout, lse, rope_base, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream);
}

ne_status ne_attn_fwd_rotated(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v, int B,
                              int H, int T, int D, float scale, ne_bf16* out, float* lse,
                              void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_fwd(s, qr, kr, v, 0.f, scale, out, 0, lse, stream, Rot::kPreRotated);
}

ne_status ne_attn_bwd_rotated(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                              const ne_bf16* out, const ne_bf16* dout, const float* lse, int B,
                              int H, int T, int D, float scale, ne_bf16* dqr, ne_bf16* dkr,
                              ne_bf16* dv, void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_bwd(s, qr, kr, v, out, dout, lse, 0.f, scale, dqr, dkr, dv, workspace,
                 workspace_bytes, stream, Rot::kPreRotated);
}

ne_status ne_attn_fwd_train(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v, int B, int H,
                            int T, int D, float rope_base, float scale, ne_bf16* out, float* lse,
                            ne_bf16* qr, ne_bf16* kr, void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_fwd(s, q, k, v, rope_base, scale, out, 0, lse, stream, Rot::kTrain, qr, kr);
}

ne_status ne_attn_bwd_train(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                            const ne_bf16* out, const ne_bf16* dout, const float* lse, int B,
                            int H, int T, int D, float rope_base, float scale, ne_bf16* dq,
                            ne_bf16* dk, ne_bf16* dv, void* workspace, size_t workspace_bytes,
                            void* stream) {
  Shape s;
  s.nseq = B;
  s.max_len = T;
  s.n_tot = (B > 0 && T > 0) ? B * T : 0;
  s.H = H;
  s.D = D;
  if (B > 0 && T > 0 && static_cast<long long>(B) * T > (1LL << 31) - 1) return NE_ERR_INVALID_ARG;
  return run_bwd(s, qr, kr, v, out, dout, lse, rope_base, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream, Rot::kTrain);
}

ne_status ne_attn_varlen_fwd_train(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                                   const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                   int H, int D, float rope_base, float scale, ne_bf16* out,
                                   float* lse, ne_bf16* qr, ne_bf16* kr, void* stream) {
  Shape s;
  s.cu = cu_seqlens;
  s.fixed = false;
  s.nseq = nseq;
  s.n_tot = n_tot;
  s.max_len = max_seqlen;
  s.H = H;
  s.D = D;
  return run_fwd(s, q, k, v, rope_base, scale, out, 0, lse, stream, Rot::kTrain, qr, kr);
}

ne_status ne_attn_varlen_bwd_train(const ne_bf16* qr, const ne_bf16* kr, const ne_bf16* v,
                                   const ne_bf16* out, const ne_bf16* dout, const float* lse,
                                   const int* cu_seqlens, int nseq, int n_tot, int max_seqlen,
                                   int H, int D, float rope_base, float scale, ne_bf16* dq,
                                   ne_bf16* dk, ne_bf16* dv, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  Shape s;
  s.cu = cu_seqlens;
  s.fixed = false;
  s.nseq = nseq;
  s.n_tot = n_tot;
  s.max_len = max_seqlen;
  s.H = H;
  s.D = D;
  return run_bwd(s, qr, kr, v, out, dout, lse, rope_base, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream, Rot::kTrain);
}

ne_status ne_attn_varlen_bwd(const ne_bf16* q, const ne_bf16* k, const ne_bf16* v,
                             const ne_bf16* out, const ne_bf16* dout, const float* lse,
                             const int* cu_seqlens, int nseq, int n_tot, int max_seqlen, int H,
                             int D, float rope_base, float scale, ne_bf16* dq, ne_bf16* dk,
                             ne_bf16* dv, void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  s.cu = cu_seqlens;
  s.fixed = false;
  s.nseq = nseq;
  s.n_tot = n_tot;
  s.max_len = max_seqlen;
  s.H = H;
  s.D = D;
  return run_bwd(s, q, k, v, out, dout, lse, rope_base, scale, dq, dk, dv, workspace,
                 workspace_bytes, stream);
}

size_t ne_attn_decode_workspace_bytes(int B, int H, int Tmax) {
  if (B <= 0 || H <= 0 || Tmax <= 0) return 0;
  return ne::decode_part_bytes(B, H, Tmax);
}

namespace {

// Shared body of the two decode entry points.  rot: q and the cached keys are
// un-rotated and rotated in the kernel; otherwise both arrive rotated (q', k').
ne_status run_decode(const ne_bf16* q, const ne_bf16* k_cache, const ne_bf16* v_cache,
                     const int* pos, int B, int H, int Tmax, int D, bool rot, float rope_base,
                     float scale, ne_bf16* out, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !pos || !out || !lse) return NE_ERR_INVALID_ARG;
  if (D != 64) return NE_ERR_UNSUPPORTED;
  if (B <= 0 || H <= 0 || Tmax <= 0) return NE_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * Tmax > 0x7fffffffLL) return NE_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale <= 0.f) return NE_ERR_INVALID_ARG;
  if (rot && (!std::isfinite(rope_base) || rope_base <= 0.f)) return NE_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(pos) ||
      !aligned4(out) || !aligned4(lse))
    return NE_ERR_MISALIGNED;
  const size_t need = ne::decode_part_bytes(B, H, Tmax);
  if (workspace && workspace_bytes < need) return NE_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15u)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  RopeTable rope{};
  CUtensorMap tt{};  // the RoPE table, 32-row boxes of half rows (unused without rotation)
  if (rot) {
    if ((rc = rope_table(*st, rope_base, Tmax, static_cast<cudaStream_t>(stream), &rope)) !=
        NE_OK)
      return rc;
    if ((rc = encode_table(&tt, rope.cs, rope.capacity, ne::kDecodeBoxRows)) != NE_OK) return rc;
  }
  CUtensorMap tk, tv;  // the caches as [B * Tmax, H, 64], 32-row boxes
  if ((rc = encode_rows(&tk, k_cache, B * Tmax, H, ne::kDecodeBoxRows)) != NE_OK) return rc;
  if ((rc = encode_rows(&tv, v_cache, B * Tmax, H, ne::kDecodeBoxRows)) != NE_OK) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  bool owned = false;
  if (!ws) {
    cudaError_t e = cudaMallocAsync(&ws, need, cs);
    if (e != cudaSuccess) return cuda_status(e);
    owned = true;
  }
  cudaError_t e = ne::launch_decode(
      tk, tv, tt, reinterpret_cast<const __nv_bfloat16*>(q), pos, B, H, Tmax, rope,
      scale * 1.4426950408889634f, static_cast<float*>(ws), reinterpret_cast<__nv_bfloat16*>(out),
      lse, st->status, cs, rot);
  if (owned) {
    cudaError_t e2 = cudaFreeAsync(ws, cs);
    if (e == cudaSuccess) e = e2;
  }
  return cuda_status(e);
}

}  // namespace

ne_status ne_attn_decode(const ne_bf16* q, const ne_bf16* k_cache, const ne_bf16* v_cache,
                         const int* pos, int B, int H, int Tmax, int D, float rope_base,
                         float scale, ne_bf16* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return run_decode(q, k_cache, v_cache, pos, B, H, Tmax, D, true, rope_base, scale, out, lse,
                    workspace, workspace_bytes, stream);
}

ne_status ne_attn_decode_rotated(const ne_bf16* qr, const ne_bf16* kr_cache,
                                 const ne_bf16* v_cache, const int* pos, int B, int H, int Tmax,
                                 int D, float scale, ne_bf16* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return run_decode(qr, kr_cache, v_cache, pos, B, H, Tmax, D, false, 0.f, scale, out, lse,
                    workspace, workspace_bytes, stream);
}

ne_status ne_rmsnorm_qkv_rope(const ne_bf16* x, const ne_bf16* g, const ne_bf16* w_qkv, int B,
                              int T, int H, int D, float eps, float rope_base, ne_bf16* x_norm,
                              float* rstd, ne_bf16* q, ne_bf16* k, ne_bf16* v, void* stream) {
  if (!x || !g || !w_qkv || !x_norm || !q || !k || !v) return NE_ERR_INVALID_ARG;
  if (D != 64) return NE_ERR_UNSUPPORTED;
  if (B <= 0 || T <= 0 || H <= 0) return NE_ERR_INVALID_ARG;
  const long long M = static_cast<long long>(B) * T;
  const long long C = static_cast<long long>(H) * 64;
  if (C % 256 != 0) return NE_ERR_UNSUPPORTED;  // H a multiple of 4
  if (M > (1LL << 31) - 1 || M * 3 * C > (1LL << 40)) return NE_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f || !std::isfinite(rope_base) || rope_base <= 0.f)
    return NE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(g) || !aligned16(w_qkv) || !aligned16(x_norm) ||
      !aligned16(q) || !aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(rstd) & 3u))
    return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  ne::gemm::Params p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(3 * C);
  p.K = static_cast<int>(C);
  p.n_tiles_m = static_cast<int>((M + 127) / 128);
  p.n_tiles_n = p.N / 256;
  p.C = static_cast<int>(C);
  p.T = T;
  p.status = st->status;
  if ((rc = rope_table(*st, rope_base, T, static_cast<cudaStream_t>(stream), &p.rope)) !=
      NE_OK)
    return rc;
  CUtensorMap ta, tw, tq, tk, tv;
  if ((rc = encode_mat(&ta, x_norm, M, p.K, 128)) != NE_OK) return rc;
  if ((rc = encode_mat(&tw, w_qkv, p.N, p.K, 256)) != NE_OK) return rc;
  if ((rc = encode_mat(&tq, q, M, p.C, 128)) != NE_OK) return rc;
  if ((rc = encode_mat(&tk, k, M, p.C, 128)) != NE_OK) return rc;
  if ((rc = encode_mat(&tv, v, M, p.C, 128)) != NE_OK) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = ne::launch_rmsnorm(reinterpret_cast<const __nv_bfloat16*>(x),
                                     reinterpret_cast<const __nv_bfloat16*>(g),
                                     reinterpret_cast<__nv_bfloat16*>(x_norm), rstd, p.M, p.C,
                                     eps, cs);
  if (e == cudaSuccess) e = ne::launch_gemm(ne::gemm::kQkvRope, ta, tw, tq, tk, tv, p, cs);
  return cuda_status(e);
}

ne_status ne_out_proj_residual(const ne_bf16* o, const ne_bf16* w_o, const ne_bf16* residual,
                               int N, int C, ne_bf16* y, void* stream) {
  if (!o || !w_o || !residual || !y) return NE_ERR_INVALID_ARG;
  if (N <= 0 || C <= 0) return NE_ERR_INVALID_ARG;
  if (C % 256 != 0) return NE_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * C > (1LL << 40)) return NE_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(w_o) || !aligned16(residual) || !aligned16(y))
    return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  ne::gemm::Params p;
  p.M = N;
  p.N = C;
  p.K = C;
  p.n_tiles_m = (N + 127) / 128;
  p.tile_n = ne::gemm_tile_n(ne::gemm::kResidual, N, C, st->sm_count);
  p.n_tiles_n = (C + p.tile_n - 1) / p.tile_n;
  p.C = C;
  p.T = 1;
  p.rope = RopeTable{nullptr, nullptr, 0};
  p.status = st->status;
  CUtensorMap ta, tw, ty, tr;
  if ((rc = encode_mat(&ta, o, N, C, 128)) != NE_OK) return rc;
  if ((rc = encode_mat(&tw, w_o, C, C, p.tile_n)) != NE_OK) return rc;
  if ((rc = encode_mat(&ty, y, N, C, 128)) != NE_OK) return rc;
  if ((rc = encode_mat(&tr, residual, N, C, 128)) != NE_OK) return rc;
  return cuda_status(
      ne::launch_gemm(ne::gemm::kResidual, ta, tw, ty, tr, tr, p, static_cast<cudaStream_t>(stream)));
}

size_t ne_mtp_head_workspace_bytes(int M, int K, int V) {
  if (M <= 0 || K <= 0 || V <= 0) return 0;
  const size_t dl = (static_cast<size_t>(M) * K * V * 2 + 255) & ~static_cast<size_t>(255);
  return dl + 256;  // dlogits bf16 [M, K*V], then the two fp32 accumulators
}

ne_status ne_mtp_head(const ne_bf16* h, const ne_bf16* w, const int* targets, int M, int C, int K,
                      int V, float* loss, float* row_loss, ne_bf16* dh, float* dw,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !w || !targets || !loss || !row_loss || !dh || !dw) return NE_ERR_INVALID_ARG;
  if (M <= 0 || C <= 0 || K <= 0 || V <= 0) return NE_ERR_INVALID_ARG;
  if (V != 256 || C % 8 != 0) return NE_ERR_UNSUPPORTED;
  if (static_cast<long long>(M) * K * V > (1LL << 40) || static_cast<long long>(M) * C > (1LL << 40) ||
      static_cast<long long>(K) * V * C > (1LL << 31))
    return NE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w) || !aligned16(dh) || !aligned16(dw) || !aligned4(targets) ||
      !aligned4(loss) || !aligned4(row_loss))
    return NE_ERR_MISALIGNED;
  const size_t need = ne_mtp_head_workspace_bytes(M, K, V);
  if (workspace && workspace_bytes < need) return NE_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  bool owned = false;
  if (!ws) {
    const cudaError_t e = cudaMallocAsync(&ws, need, cs);
    if (e != cudaSuccess) return cuda_status(e);
    owned = true;
  }
  const int N = K * V;
  ne_bf16* dlogits = static_cast<ne_bf16*>(ws);
  float* acc = reinterpret_cast<float*>(static_cast<char*>(ws) + need - 256);
  // 1. logits = h . W^T with the cross-entropy epilogue -> dlogits, row losses, sums
  ne::gemm::Params p1;
  p1.M = M;
  p1.N = N;
  p1.K = C;
  p1.n_tiles_m = (M + 127) / 128;
  p1.n_tiles_n = K;
  p1.targets = targets;
  p1.heads = K;
  p1.row_loss = row_loss;
  p1.acc = acc;
  p1.status = st->status;
  // 2. dh = dlogits . W / n (W read MN-major: its rows are the contraction)
  ne::gemm::Params p2;
  p2.M = M;
  p2.N = C;
  p2.K = N;
  p2.n_tiles_m = (M + 127) / 128;
  p2.tile_n = ne::gemm_tile_n(ne::gemm::kScale, M, C, st->sm_count);
  p2.n_tiles_n = (C + p2.tile_n - 1) / p2.tile_n;
  p2.acc = acc;
  p2.loss = loss;
  p2.status = st->status;
  // 3. dW = dlogits^T . h / n, both read MN-major, the tokens split over the
  // CTAs (partial tiles reduce-added in fp32)
  ne::gemm::Params p3;
  p3.M = N;
  p3.N = C;
  p3.K = M;
  p3.n_tiles_m = (N + 127) / 128;
  p3.n_tiles_n = (C + 255) / 256;
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 148;
    const int k_chunks = (M + 63) / 64;
    const int n_mn = p3.n_tiles_m * p3.n_tiles_n;
    int splits = sms / n_mn;
    splits = splits < 1 ? 1 : (splits > k_chunks ? k_chunks : splits);
    p3.chunks_per_split = (k_chunks + splits - 1) / splits;
    p3.k_splits = (k_chunks + p3.chunks_per_split - 1) / p3.chunks_per_split;  // none empty
  }
  p3.acc = acc;
  p3.status = st->status;
  CUtensorMap th_k, tw_k, tdl_k, tw_mn, tdh, tdl_mn, th_mn, tdw;
  if ((rc = encode_mat(&th_k, h, M, C, 128)) == NE_OK &&
      (rc = encode_mat(&tw_k, w, N, C, 256)) == NE_OK &&
      (rc = encode_mat(&tdl_k, dlogits, M, N, 128)) == NE_OK &&
      (rc = encode_mat(&tw_mn, w, N, C, 64)) == NE_OK &&
      (rc = encode_mat(&tdh, dh, M, C, 128)) == NE_OK &&
      (rc = encode_mat(&tdl_mn, dlogits, M, N, 64)) == NE_OK &&
      (rc = encode_mat(&th_mn, h, M, C, 64)) == NE_OK)
    rc = encode_mat_f32(&tdw, dw, N, C, 128);
  cudaError_t e = cudaSuccess;
  if (rc == NE_OK) {
    e = cudaMemsetAsync(acc, 0, 2 * sizeof(float), cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw, 0, static_cast<size_t>(N) * C * sizeof(float), cs);
    if (e == cudaSuccess)
      e = ne::launch_gemm(ne::gemm::kMtpCe, th_k, tw_k, tdl_k, tdl_k, tdl_k, p1, cs);
    if (e == cudaSuccess)
      e = ne::launch_gemm(ne::gemm::kScale, tdl_k, tw_mn, tdh, tdh, tdh, p2, cs);
    if (e == cudaSuccess)
      e = ne::launch_gemm(ne::gemm::kReduceF32, tdl_mn, th_mn, tdw, tdw, tdw, p3, cs);
  }
  if (owned) {
    const cudaError_t e2 = cudaFreeAsync(ws, cs);
    if (e == cudaSuccess) e = e2;
  }
  if (rc != NE_OK) return rc;
  return cuda_status(e);
}

ne_status ne_attn_set_bwd_phase_events(void* ev_after_preprocess, void* ev_after_main) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if ((ev_after_preprocess == nullptr) != (ev_after_main == nullptr)) return NE_ERR_INVALID_ARG;
  g_ev_pre = static_cast<cudaEvent_t>(ev_after_preprocess);
  g_ev_main = static_cast<cudaEvent_t>(ev_after_main);
  return NE_OK;
}

ne_status ne_attn_set_fwd_phase_event(void* ev_after_rotation) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_ev_rot = static_cast<cudaEvent_t>(ev_after_rotation);
  return NE_OK;
}

ne_status ne_attn_get_device_status(void* stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NE_ERR_CUDA;
  int code = 0;
  if (cudaMemcpyFromSymbol(&code, g_device_status, sizeof(int)) != cudaSuccess) return NE_ERR_CUDA;
  const int zero = 0;
  if (code != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
    return NE_ERR_CUDA;
  g_last_code = code;
  if (code == ne::NE_DEV_OK) return NE_OK;
  if (code == ne::NE_DEV_BAD_SEQLEN) return NE_ERR_BAD_SEQLEN;
  if (code >= ne::NE_DEV_TIMEOUT_BASE) return NE_ERR_TIMEOUT;
  return NE_ERR_CUDA;
}

int ne_attn_last_device_code(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  return g_last_code;
}

void ne_attn_release(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& st = g_dev[d];
    if (st.tables.empty() && st.retired.empty() && st.scratch.empty() && st.scheds.empty())
      continue;
    cudaSetDevice(d);
    for (auto& t : st.tables) cudaFree(t.dev);
    for (auto& e : st.scheds)
      if (e.dev) cudaFree(e.dev);
    st.scheds.clear();
    for (auto* p : st.retired) cudaFree(p);
    for (auto& e : st.scratch) cudaFreeAsync(e.ptr, e.stream);
    if (!st.scratch.empty()) cudaDeviceSynchronize();
    st.tables.clear();
    st.retired.clear();
    st.scratch.clear();
  }
  cudaSetDevice(cur);
}

// ------------------------------------------------------------ debug entries --

int ne_debug_schedule(int nseq, int H, int T, int G, int* out, int out_len) {
  if (nseq <= 0 || H <= 0 || T <= 0 || G <= 0 || !out || out_len < 0 ||
      static_cast<long long>(nseq) * H * ((T + 127) / 128) > (1 << 24))
    return -1;
  const std::vector<int> tab =
      ne::pack_schedule(ne::unit_steps(nseq, H, T), G, kBwdOverhead[0], kBwdOverhead[1]);
  if (tab.size() > static_cast<size_t>(out_len)) return -1;
  std::copy(tab.begin(), tab.end(), out);
  return static_cast<int>(tab.size());
}

ne_status ne_debug_tma_tile(const ne_bf16* src, int n_rows, int H, int h, int row0,
                            void* dst_raw, void* stream) {
  if (!src || !dst_raw || n_rows <= 0 || H <= 0 || h < 0 || h >= H) return NE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst_raw)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  CUtensorMap tm;
  if ((rc = encode_rows(&tm, src, n_rows, H)) != NE_OK) return rc;
  return cuda_status(ne::launch_debug_tile(tm, h, row0, 0, 0, RopeTable{nullptr, nullptr, 0}, dst_raw,
                                           nullptr, st->status,
                                           static_cast<cudaStream_t>(stream)));
}

ne_status ne_debug_rope_tile(const ne_bf16* src, int n_rows, int H, int h, int row0, int pos0,
                             float rope_base, ne_bf16* dst, void* stream) {
  if (!src || !dst || n_rows <= 0 || H <= 0 || h < 0 || h >= H || pos0 < 0)
    return NE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return NE_ERR_MISALIGNED;
  if (!std::isfinite(rope_base) || rope_base <= 0.f) return NE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  RopeTable rt;
  if ((rc = rope_table(*st, rope_base, pos0 + 128, static_cast<cudaStream_t>(stream), &rt)) !=
      NE_OK)
    return rc;
  CUtensorMap tm;
  if ((rc = encode_rows(&tm, src, n_rows, H)) != NE_OK) return rc;
  return cuda_status(ne::launch_debug_tile(tm, h, row0, 1, pos0, rt, nullptr,
                                           reinterpret_cast<__nv_bfloat16*>(dst), st->status,
                                           static_cast<cudaStream_t>(stream)));
}

ne_status ne_debug_umma(int form, const ne_bf16* a, const ne_bf16* b, float* d, void* stream) {
  if (form < 0 || form > 3 || !a || !b || !d) return NE_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  return cuda_status(ne::launch_debug_umma(form, reinterpret_cast<const __nv_bfloat16*>(a),
                                           reinterpret_cast<const __nv_bfloat16*>(b), d,
                                           st->status, static_cast<cudaStream_t>(stream)));
}

ne_status ne_debug_pipeline(const ne_bf16* src, int n_rows, int H, int n_items, int drop_item,
                            long long wait_limit_cycles, float* d, void* stream) {
  if (!src || !d || n_rows <= 0 || H <= 0 || n_items < 1 || n_items > 64 ||
      static_cast<long long>(n_items) * 128 > n_rows || drop_item < -1 || drop_item >= n_items ||
      wait_limit_cycles < 1000 || wait_limit_cycles > 2000000000LL)
    return NE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(d)) return NE_ERR_MISALIGNED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  ne_status rc = device_state(&st);
  if (rc != NE_OK) return rc;
  if ((rc = get_encoder()) != NE_OK) return rc;
  CUtensorMap tm;
  if ((rc = encode_rows(&tm, src, n_rows, H)) != NE_OK) return rc;
  return cuda_status(ne::launch_debug_pipeline(tm, n_items, drop_item, wait_limit_cycles, d,
                                               st->status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
