// ne_attn_decode.cu -- decode attention over a KV cache with RoPE, sm_103a.
//
// Generation adds one token at a time (the interactive text generation of the
// NanoEuler Show HN page and of "Tiny Hackable CUDA", section 7): the new
// query at position m attends to the cached keys and values at positions
// 0..m, with the same RoPE and softmax as the training forward:
//   o = sum_{n<=m} softmax_n(scale * q'_m . k'_n) v_n,   q' = R(m) q, k' = R(n) k.
// Every cached key is read once per step, so the operation is bound by HBM
// bandwidth; it runs on the CUDA cores (one query row is a matrix-vector
// product, nothing for the tensor cores to share).
//
// Two kernels on one stream:
//   1. split: one CTA per (chunk of keys, head, sequence) -- 1024 keys when
//      that still gives a few waves of CTAs, else 256.  Warp 8 streams the
//      chunk through a shared-memory ring with TMA: per stage the K
//      and V boxes of 32 consecutive positions (4 KiB each) and the 32 rows
//      of the RoPE table as two boxes of half rows (4 KiB each), all with the
//      128-byte swizzle, so that the warps' reads spread over the banks (the
//      table rows read contiguously made 8-way bank conflicts).  Warps 0-7
//      take 4 keys of each stage; eight lanes share one 128-byte key row,
//      lane c holding dims 4c .. 4c + 3 and their RoPE partners 32 + 4c ..
//      32 + 4c + 3, so that it rotates its own dims with one read of the 4
//      (cos, sin) pairs they share (an earlier layout, 16 contiguous bytes
//      per lane, read every table pair twice and fetched the partner dims by
//      shuffles: 3.99-4.16 TB/s).  A group of eight lanes keeps its own
//      online softmax (max, sum, its 8 output dims); groups, then warps,
//      are merged and the CTA writes one partial (m, l, o[64]).
//      Three CTAs per SM (24 consumer warps) measured best: 3.86 TB/s at
//      B8 H12 Tmax16384 against 2.69 with 4 warps and 8 stages -- the
//      consumers' per-key chain (swizzled loads, RoPE, dot, shuffles, exp)
//      needs the warps more than the ring needs depth.
//   2. merge: one warp per (sequence, head) combines the chunk partials with
//      their log-sum-exp weights into o (bf16) and LSE (fp32, natural log).
// Keys are rotated with the fp32 rule of the training kernels and rounded to
// bf16, so a decode at position T-1 sees exactly the operands the training
// forward multiplies.  kRot = false: the caller passes q' and a cache of
// rotated keys k' (as the training forward or the QKV projection with RoPE
// writes them); nothing is rotated, no table rows are loaded, and a ring
// of 4 stages holds only the K and V boxes (5 CTAs per SM).
#include "ne_sm100.cuh"

namespace ne {

namespace dec {
constexpr int kChunkUnit = 256;      // keys per CTA are a multiple of this
constexpr int kWarps = 8;            // consumer warps: a stage's 32 keys, 4 per warp
constexpr int kThreads = (kWarps + 1) * 32;  // + the TMA producer warp
constexpr int kKeys = 32;            // keys per stage (the TMA box height)
constexpr int kKvBytes = kKeys * 128;                  // one K or V box
constexpr int kTabBytes = kKeys * 256;                 // 16 table rows
// Shared memory of each instantiation: the ring (K, V and, when keys are
// rotated here, the table rows), barriers, the warps' partial states.
template <bool kRot>
struct Smem {
  // Ring depth: 3 stages of 16 KiB when keys are rotated here; 4 of 8 KiB on
  // a cache of rotated keys (measured on decode16k: 3 % faster than 3, still
  // 5 CTAs per SM).
  static constexpr int kStages = kRot ? 3 : 4;
  static constexpr int kStageBytes = 2 * kKvBytes + (kRot ? kTabBytes : 0);  // 16 / 8 KiB
  static constexpr int OFF_BAR = kStages * kStageBytes;
  static constexpr int OFF_RED = OFF_BAR + 2 * kStages * 8 + 16;
  static constexpr int BYTES = OFF_RED + kWarps * 66 * 4 + 1024;  // + slack for 1024-byte alignment
};
constexpr int kPartFloats = 68;      // m, l, 2 pad, o[64] (16-byte multiple)
}  // namespace dec

// Lane c (0..7) of a key's lane group holds the 8 dims {4c .. 4c + 3} and
// their RoPE partners {32 + 4c .. 32 + 4c + 3}, as 4 packed fp32 pairs: [0], [1]
// the low quad, [2], [3] the high quad.  A lane then rotates its own dims
// with the 4 (cos, sin) pairs of frequencies 4c .. 4c + 3 (two float4s) and
// no partner exchange.

// bf16 words (lo, hi quad: 8 bytes each) -> 4 packed fp32 pairs.
__device__ __forceinline__ void unpack_quads(uint2 lo, uint2 hi, uint64_t (&x)[4]) {
  x[0] = f2_pack(bf16lo_to_f32(lo.x), bf16hi_to_f32(lo.x));
  x[1] = f2_pack(bf16lo_to_f32(lo.y), bf16hi_to_f32(lo.y));
  x[2] = f2_pack(bf16lo_to_f32(hi.x), bf16hi_to_f32(hi.x));
  x[3] = f2_pack(bf16lo_to_f32(hi.y), bf16hi_to_f32(hi.y));
}

// Rotate a lane's 8 dims with the fp32 rule of the training kernels: dim i of
// the low half gets fma(x_i, cos, -(x_{i+32} sin)), dim i + 32 gets
// fma(x_{i+32}, cos, x_i sin) (x (-sin) is exactly -(x sin)); each result is
// rounded to bf16 and kept as fp32.  t[0], t[1]: (cos, sin, cos, sin) of
// frequencies 4c, 4c + 1 and 4c + 2, 4c + 3.
__device__ __forceinline__ void rope_quads(const uint64_t (&x)[4], const float4 (&t)[2],
                                           uint64_t (&out)[4]) {
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint64_t cs = f2_pack(t[u].x, t[u].z);
    const uint64_t sn = f2_pack(t[u].y, t[u].w);
    const uint64_t nsn = f2_pack(-t[u].y, -t[u].w);
    float a0, a1, b0, b1;
    f2_unpack(f2_fma(x[u], cs, f2_mul(x[u + 2], nsn)), a0, a1);
    f2_unpack(f2_fma(x[u + 2], cs, f2_mul(x[u], sn)), b0, b1);
    const uint32_t ha = pack_bf16x2(a0, a1), hb = pack_bf16x2(b0, b1);  // round to nearest even
    out[u] = f2_pack(bf16lo_to_f32(ha), bf16hi_to_f32(ha));
    out[u + 2] = f2_pack(bf16lo_to_f32(hb), bf16hi_to_f32(hb));
  }
}

// A lane's two quads of a 128-byte-swizzled 64-dim bf16 row in shared memory.
// Lane groups of odd index load the high quad first, so that the 4 rows one
// warp instruction touches fall half on each half of the banks.
__device__ __forceinline__ void load_quads(const uint8_t* base, int row, int c, int grp,
                                           uint2& lo, uint2& hi) {
  const int first = grp & 1;  // 0: low quad first
  const uint32_t in = (c & 1) * 8;
  const uint2 a = *reinterpret_cast<const uint2*>(base + sw128_offset(row, 4 * first + (c >> 1)) + in);
  const uint2 b = *reinterpret_cast<const uint2*>(base + sw128_offset(row, 4 * (first ^ 1) + (c >> 1)) + in);
  lo = first ? b : a;
  hi = first ? a : b;
}

// The (cos, sin) pairs of frequencies 4c .. 4c + 3 of a stage's table row:
// half c >> 2 of the row (pairs 16 (c >> 2) ..), 16-byte units 2 (c & 3) and
// 2 (c & 3) + 1 of that half.  Lanes of the second half take their units in
// the other order, so that one instruction reads even units of one half and
// odd units of the other (no two lanes of a row on the same banks).
__device__ __forceinline__ void load_table_quads(const uint8_t* halves, int row, int c,
                                                 float4 (&t)[2]) {
  const int sw = c >> 2;
  const uint8_t* h = halves + sw * dec::kKvBytes;
  const float4 a = *reinterpret_cast<const float4*>(h + sw128_offset(row, 2 * (c & 3) + sw));
  const float4 b = *reinterpret_cast<const float4*>(h + sw128_offset(row, 2 * (c & 3) + 1 - sw));
  t[0] = sw ? b : a;
  t[1] = sw ? a : b;
}

// Merge online-softmax state (m, l, o[8]) with another (log2 units).
__device__ __forceinline__ void merge_state(float& m, float& l, float (&o)[8], float m2, float l2,
                                            const float (&o2)[8]) {
  const float mn = fmaxf(m, m2);
  const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
  const float b = (m2 == -INFINITY) ? 0.f : ex2_approx(m2 - mn);
  l = l * a + l2 * b;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = o[e] * a + o2[e] * b;
  m = mn;
}

// Registers: the rotating instantiation is left free (70 per thread: its
// per-key chain of table reads, rotation and dot keeps more values live; with
// the compiler's default 52 it ran 8% slower on decode16k); the other is held
// to 5 CTAs per SM (40 per thread).
template <bool kRot>
__global__ void __launch_bounds__(dec::kThreads, kRot ? 1 : 5)
    ne_attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV,
                                const __grid_constant__ CUtensorMap tmT,
                                const __nv_bfloat16* __restrict__ q, const int* __restrict__ pos,
                                int H, int Tmax, RopeTable rope, float scale_log2,
                                float* __restrict__ part, int chunk, int n_chunks, int* status) {
  using namespace dec;
  using L = Smem<kRot>;
  constexpr int kStageBytes = L::kStageBytes;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 2 * kStages * 8);
  float (*red)[66] = reinterpret_cast<float (*)[66]>(smem + L::OFF_RED);

  // Heads vary fastest over the grid: the CTAs running together read the
  // 12 neighbouring 128-byte pieces of the same cache rows.
  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cl = lane & 7;   // this lane's dims: 4cl..4cl+3 and 32+4cl..32+4cl+3
  const int grp = lane >> 3; // which of the warp's 4 keys per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // Launched with programmatic dependent launch: the set-up above overlaps the
  // previous kernel on the stream (e.g. the one that appended to the cache).
  pdl_wait();
  pdl_launch_dependents();

  const int m_pos = __ldg(pos + b);
  const bool bad = (m_pos < 0 || m_pos >= Tmax);
  if (bad && c == 0 && h == 0 && threadIdx.x == 0 && status) atomicCAS(status, 0, NE_DEV_BAD_SEQLEN);
  const int n_keys = bad ? 0 : m_pos + 1;
  const int kbeg = c * chunk;
  const int k_end = min(kbeg + chunk, n_keys);
  const int n_st = k_end > kbeg ? (k_end - kbeg + kKeys - 1) / kKeys : 0;  // stages of this CTA

  if (warp == kWarps) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (kRot) tma_prefetch_desc(&tmT);
      int i = 0;
      for (; i < n_st; ++i) {
        const int s = i % kStages;
        if (i >= kStages &&
            !mbar_wait(&empty[s], ((i - kStages) / kStages) & 1, abort_flag, status, 50))
          break;
        uint8_t* st = smem + s * kStageBytes;
        const int key0 = kbeg + kKeys * i;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        // Rows past the cache of the last sequence (and table rows past the
        // table) are filled with zeros by the TMA unit.
        tma_load_3d(st, &tmK, &full[s], 0, h, b * Tmax + key0);
        tma_load_3d(st + kKvBytes, &tmV, &full[s], 0, h, b * Tmax + key0);
        if constexpr (kRot) {
          tma_load_2d(st + 2 * kKvBytes, &tmT, &full[s], 0, key0);
          tma_load_2d(st + 3 * kKvBytes, &tmT, &full[s], 32, key0);
        }
      }
      // Every copy issued has landed before this warp exits (on the normal
      // path the consumers have already waited for them; after an abort they
      // may not have).
      for (int j = (i > kStages ? i - kStages : 0); j < i; ++j) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&full[j % kStages], (j / kStages) & 1) &&
               clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  // q' = R(m) q, this lane's 8 dims (every lane group holds a copy).
  uint64_t q2[4];
  {
    const uint2* qrow = reinterpret_cast<const uint2*>(q + (static_cast<long long>(b) * H + h) * 64);
    uint64_t x[4];
    unpack_quads(__ldg(qrow + cl), __ldg(qrow + 8 + cl), x);
    if constexpr (kRot) {
      const float4* tq = reinterpret_cast<const float4*>(
          rope.cs + static_cast<long long>(bad ? 0 : m_pos) * 32 + 4 * cl);
      const float4 t[2] = {__ldg(tq), __ldg(tq + 1)};
      rope_quads(x, t, q2);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) q2[u] = x[u];
    }
  }

  // Online softmax of each lane group against a reference max m_ref (log2
  // units) that moves only when a score exceeds it by more than 2^8 (exact:
  // o and l keep a common reference, so the usual rescale of every key is
  // skipped); o as 4 packed pairs.
  float m_ref = -INFINITY, l = 0.f;
  uint64_t o2[4] = {0, 0, 0, 0};
  const int row = 4 * warp + grp;  // this lane group's row of every stage
  bool ok = true;
  for (int i = 0; ok && i < n_st; ++i) {
    const int s = i % kStages;
    if (!(ok = mbar_wait_warp(&full[s], (i / kStages) & 1, abort_flag, status, 51))) break;
    const uint8_t* st = smem + s * kStageBytes;
    uint2 klo, khi, vlo, vhi;
    load_quads(st, row, cl, grp, klo, khi);
    load_quads(st + kKvBytes, row, cl, grp, vlo, vhi);
    const bool live = kbeg + kKeys * i + row < k_end;
    uint64_t k2[4];
    if constexpr (kRot) {
      float4 tb[2];
      load_table_quads(st + 2 * kKvBytes, row, cl, tb);
      uint64_t x[4];
      unpack_quads(klo, khi, x);
      rope_quads(x, tb, k2);
    } else {
      unpack_quads(klo, khi, k2);
    }
    uint64_t d2 = f2_mul(q2[0], k2[0]);
#pragma unroll
    for (int u = 1; u < 4; ++u) d2 = f2_fma(q2[u], k2[u], d2);
    float d0, d1;
    f2_unpack(d2, d0, d1);
    float dot = d0 + d1;
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    dot += __shfl_xor_sync(0xffffffffu, dot, 4);
    uint64_t v2[4];
    unpack_quads(vlo, vhi, v2);
    // Every value read from the stage is in registers now: release it.
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (live) {
      const float sc = dot * scale_log2;
      if (sc > m_ref + 8.f) {  // also the group's first key (m_ref = -inf)
        const float a = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - sc);
        const uint64_t a2 = f2_pack(a, a);
        l *= a;
#pragma unroll
        for (int u = 0; u < 4; ++u) o2[u] = f2_mul(o2[u], a2);
        m_ref = sc;
      }
      const float pk = ex2_approx(sc - m_ref);
      const uint64_t p2 = f2_pack(pk, pk);
      l += pk;
#pragma unroll
      for (int u = 0; u < 4; ++u) o2[u] = f2_fma(p2, v2[u], o2[u]);
    }
  }
  float m = m_ref, o[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) f2_unpack(o2[u], o[2 * u], o[2 * u + 1]);
  // Merge the 4 lane groups (lanes cl, cl + 8, cl + 16, cl + 24).
#pragma unroll
  for (int sh = 8; sh <= 16; sh <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, sh);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, sh);
    float o2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, o[e], sh);
    merge_state(m, l, o, m2, l2, o2);
  }
  if (lane < 8) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      red[warp][2 + 4 * cl + e] = o[e];
      red[warp][2 + 32 + 4 * cl + e] = o[4 + e];
    }
    if (lane == 0) {
      red[warp][0] = m;
      red[warp][1] = l;
    }
  }
  named_bar_sync(1, kWarps * 32);  // the consumer warps only
  // Merge the warps: thread t < 64 owns output dim t.
  float* dst = part + ((static_cast<long long>(b) * H + h) * n_chunks + c) * kPartFloats;
  if (threadIdx.x < 64) {
    const int d = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[w][0]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red[w][0];
      const float a = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      L += red[w][1] * a;
      O += red[w][2 + d] * a;
    }
    dst[4 + d] = O;
    if (d == 0) {
      dst[0] = M;
      dst[1] = L;
    }
  }
}

__global__ void __launch_bounds__(32)
    ne_attn_decode_merge_kernel(const float* __restrict__ part, int n_chunks,
                                __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  using namespace dec;
  pdl_wait();  // the split kernel's partials are complete
  pdl_launch_dependents();
  const long long bh = blockIdx.x;
  const int lane = threadIdx.x;
  const float* src = part + bh * n_chunks * kPartFloats;
  // Lane c holds chunk c's (m, l) (chunks past 32 fold in by lane stride);
  // an empty chunk has m = -inf, l = 0 and a zero partial output.
  float M = -INFINITY;
  for (int c = lane; c < n_chunks; c += 32) M = fmaxf(M, src[c * kPartFloats]);
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
  float L = 0.f, o0 = 0.f, o1 = 0.f;  // lane owns dims 2*lane, 2*lane + 1
  for (int c0 = 0; c0 < n_chunks; c0 += 32) {
    const int c = c0 + lane;
    float w = 0.f, lw = 0.f;
    if (c < n_chunks) {
      const float mc = src[c * kPartFloats];
      w = (mc == -INFINITY) ? 0.f : ex2_approx(mc - M);
      lw = src[c * kPartFloats + 1] * w;
    }
    L += lw;
    const int nc = min(32, n_chunks - c0);
    for (int j = 0; j < nc; ++j) {  // weights from lane j; loads independent of each other
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const float2 oc = reinterpret_cast<const float2*>(src + (c0 + j) * kPartFloats + 4)[lane];
      o0 = __fmaf_rn(oc.x, wj, o0);
      o1 = __fmaf_rn(oc.y, wj, o1);
    }
  }
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) L += __shfl_xor_sync(0xffffffffu, L, sh);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  reinterpret_cast<uint32_t*>(out + bh * 64)[lane] = pack_bf16x2(o0 * inv, o1 * inv);
  if (lane == 0) lse[bh] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

int decode_chunks(int Tmax) { return (Tmax + dec::kChunkUnit - 1) / dec::kChunkUnit; }

size_t decode_part_bytes(int B, int H, int Tmax) {
  return static_cast<size_t>(B) * H * decode_chunks(Tmax) * dec::kPartFloats * sizeof(float);
}

// rot: q and the cached keys are rotated here (tmT: the table); otherwise the
// caller passed q' and a cache of k' (tmT unused).
cudaError_t launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmT,
                          const __nv_bfloat16* q, const int* pos, int B, int H, int Tmax,
                          const RopeTable& rope, float scale_log2, float* part,
                          __nv_bfloat16* out, float* lse, int* status, cudaStream_t stream,
                          bool rot) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_attn_decode_split_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         dec::Smem<true>::BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ne_attn_decode_split_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, dec::Smem<false>::BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // 1024 keys per CTA when that still leaves a few waves of CTAs (each CTA's
  // set-up, pipeline fill and merge are then spread over more keys).
  const long long big = static_cast<long long>(B) * H * ((Tmax + 1023) / 1024);
  const int chunk = big >= 1024 ? 1024 : dec::kChunkUnit;
  const int n_chunks = (Tmax + chunk - 1) / chunk;
  dim3 grid(H, n_chunks, B);
  cudaError_t e =
      rot ? launch_pdl(ne_attn_decode_split_kernel<true>, grid, dim3(dec::kThreads),
                       dec::Smem<true>::BYTES, stream, tmK, tmV, tmT, q, pos, H, Tmax, rope,
                       scale_log2, part, chunk, n_chunks, status)
          : launch_pdl(ne_attn_decode_split_kernel<false>, grid, dim3(dec::kThreads),
                       dec::Smem<false>::BYTES, stream, tmK, tmV, tmT, q, pos, H, Tmax, rope,
                       scale_log2, part, chunk, n_chunks, status);
  if (e != cudaSuccess) return e;
  return launch_pdl(ne_attn_decode_merge_kernel, dim3(B * H), dim3(32), 0, stream, part, n_chunks,
                    out, lse);
}

}  // namespace ne
