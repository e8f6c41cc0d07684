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
//      take 4 keys of each stage; eight lanes share one 128-byte key row
//      (lane l: chunk l % 8, 16 bytes), its RoPE partner chunk comes from
//      lane l ^ 4 by a shuffle.  A group of eight lanes keeps its own online
//      softmax (max, sum, the 8 output dims of its chunk); groups, then
//      warps, are merged and the CTA writes one partial (m, l, o[64]).
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
// of 4 stages holds only the K and V boxes (40 registers, 5 CTAs per SM).
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

// The 8 (cos, sin) pairs of the dims of chunk c (dims 8(c & 3) .. + 7 of the
// 32 frequencies) of table row `cs` (one position), as 4 float4.
__device__ __forceinline__ void load_pairs(const float2* __restrict__ cs, int c, float4 (&t)[4]) {
  const float4* p = reinterpret_cast<const float4*>(cs + 8 * (c & 3));
#pragma unroll
  for (int u = 0; u < 4; ++u) t[u] = __ldg(p + u);
}

// The 8 bf16 dims of a 16-byte chunk as 4 packed fp32 pairs.
__device__ __forceinline__ void unpack8x2(const uint4 w, uint64_t (&x)[4]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = f2_pack(bf16lo_to_f32(u[e]), bf16hi_to_f32(u[e]));
}

// Rotate the 8 dims of chunk c (dims 8c..8c+7 of a 64-dim row) given the 8
// dims of its partner chunk c ^ 4 and the chunk's (cos, sin) pairs, two dims
// per packed instruction; the result is rounded to bf16 and returned as fp32
// pairs.  c < 4: x holds element i, y element i + 32, x' = fma(x, cos,
// -(y sin)); c >= 4: x holds element i + 32, y element i, x' = fma(x, cos,
// y sin).  The sign is folded into sin: y (-sin) is exactly -(y sin).
__device__ __forceinline__ void rope_chunk2(const uint64_t (&x)[4], const uint64_t (&y)[4], int c,
                                            const float4 (&t)[4], uint64_t (&out)[4]) {
  const float sg = (c < 4) ? -1.f : 1.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint64_t cs = f2_pack(t[u].x, t[u].z);
    const uint64_t sn = f2_pack(sg * t[u].y, sg * t[u].w);
    float r0, r1;
    f2_unpack(f2_fma(x[u], cs, f2_mul(y[u], sn)), r0, r1);
    const uint32_t h = pack_bf16x2(r0, r1);  // round to nearest even
    out[u] = f2_pack(bf16lo_to_f32(h), bf16hi_to_f32(h));
  }
}

__device__ __forceinline__ uint4 shfl_xor_u4(uint4 w, int m) {
  w.x = __shfl_xor_sync(0xffffffffu, w.x, m);
  w.y = __shfl_xor_sync(0xffffffffu, w.y, m);
  w.z = __shfl_xor_sync(0xffffffffu, w.z, m);
  w.w = __shfl_xor_sync(0xffffffffu, w.w, m);
  return w;
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

template <bool kRot>
__global__ void __launch_bounds__(dec::kThreads)
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
  const int cl = lane & 7;   // 16-byte chunk of the row this lane holds
  const int grp = lane >> 3; // which of the warp's 4 keys per stage

  const int m_pos = __ldg(pos + b);
  const bool bad = (m_pos < 0 || m_pos >= Tmax);
  if (bad && c == 0 && h == 0 && threadIdx.x == 0 && status) atomicCAS(status, 0, NE_DEV_BAD_SEQLEN);
  const int n_keys = bad ? 0 : m_pos + 1;
  const int kbeg = c * chunk;
  const int k_end = min(kbeg + chunk, n_keys);
  const int n_st = k_end > kbeg ? (k_end - kbeg + kKeys - 1) / kKeys : 0;  // stages of this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

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
  // q' = R(m) q, the 8 dims of chunk cl (every lane group holds a copy).
  uint64_t q2[4];
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(q + (static_cast<long long>(b) * H + h) * 64);
    const uint4 w = __ldg(qrow + cl);
    if constexpr (kRot) {
      uint64_t x[4], y[4];
      float4 t[4];
      load_pairs(rope.cs + static_cast<long long>(bad ? 0 : m_pos) * 32, cl, t);
      unpack8x2(w, x);
      unpack8x2(shfl_xor_u4(w, 4), y);
      rope_chunk2(x, y, cl, t, q2);
    } else {
      unpack8x2(w, q2);
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
    const uint4 wk = *reinterpret_cast<const uint4*>(st + sw128_offset(row, cl));
    const uint4 wv = *reinterpret_cast<const uint4*>(st + kKvBytes + sw128_offset(row, cl));
    const bool live = kbeg + kKeys * i + row < k_end;
    uint64_t k2[4];
    if constexpr (kRot) {
      float4 tb[4];
      // Pairs 8q .. 8q + 7 (q = cl & 3): half q >> 1 of the row, 16-byte
      // units 4 (q & 1) .. + 3 of that half, swizzled like K and V.
      const uint8_t* half = st + (2 + ((cl & 3) >> 1)) * kKvBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        tb[u] = *reinterpret_cast<const float4*>(half + sw128_offset(row, 4 * (cl & 1) + u));
      uint64_t x[4], y[4];
      unpack8x2(wk, x);
      unpack8x2(shfl_xor_u4(wk, 4), y);
      rope_chunk2(x, y, cl, tb, k2);
    } else {
      unpack8x2(wk, k2);
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
    unpack8x2(wv, v2);
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
    for (int e = 0; e < 8; ++e) red[warp][2 + 8 * cl + e] = o[e];
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
  if (rot)
    ne_attn_decode_split_kernel<true><<<grid, dec::kThreads, dec::Smem<true>::BYTES, stream>>>(
        tmK, tmV, tmT, q, pos, H, Tmax, rope, scale_log2, part, chunk, n_chunks, status);
  else
    ne_attn_decode_split_kernel<false><<<grid, dec::kThreads, dec::Smem<false>::BYTES, stream>>>(
        tmK, tmV, tmT, q, pos, H, Tmax, rope, scale_log2, part, chunk, n_chunks, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ne_attn_decode_merge_kernel<<<B * H, 32, 0, stream>>>(part, n_chunks, out, lse);
  return cudaGetLastError();
}

}  // namespace ne
