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
//   1. split: one CTA per (256-key chunk, head, sequence).  Each round the
//      CTA's 4 warps take 16 consecutive keys, 4 per warp; eight lanes share
//      one 128-byte key row (lane l: chunk l % 8, 16 bytes), its RoPE partner
//      chunk comes from lane l ^ 4 by a shuffle.  A
//      group of eight lanes keeps its own online softmax (max, sum, the 8
//      output dims of its chunk); groups, then warps, are merged and the CTA
//      writes one partial (m, l, o[64]) of its chunk.
//   2. merge: one warp per (sequence, head) combines the chunk partials with
//      their log-sum-exp weights into o (bf16) and LSE (fp32, natural log).
// Keys are rotated with the fp32 rule of the training kernels and rounded to
// bf16, so a decode at position T-1 sees exactly the operands the training
// forward multiplies.
#include "ne_sm100.cuh"

namespace ne {

namespace dec {
constexpr int kChunkUnit = 256;      // keys per CTA are a multiple of this
constexpr int kWarps = 4;            // a round covers 16 consecutive keys: 4 per warp
constexpr int kPartFloats = 68;      // m, l, 2 pad, o[64] (16-byte multiple)
}  // namespace dec

// The 8 (cos, sin) pairs of the dims of chunk c (dims 8(c & 3) .. + 7 of the
// 32 frequencies) of table row `cs` (one position), as 4 float4.
__device__ __forceinline__ void load_pairs(const float2* __restrict__ cs, int c, float4 (&t)[4]) {
  const float4* p = reinterpret_cast<const float4*>(cs + 8 * (c & 3));
#pragma unroll
  for (int u = 0; u < 4; ++u) t[u] = __ldg(p + u);
}

// Rotate the 8 dims of chunk c (dims 8c..8c+7 of a 64-dim row) given the 8
// dims of its partner chunk c ^ 4 and the chunk's (cos, sin) pairs; the
// result is rounded to bf16 and returned as fp32.
__device__ __forceinline__ void rope_chunk(const float (&x)[8], const float (&y)[8], int c,
                                           const float4 (&t)[4], float (&out)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float cs_c = (e & 1) ? t[e >> 1].z : t[e >> 1].x;
    const float cs_s = (e & 1) ? t[e >> 1].w : t[e >> 1].y;
    // c < 4: x is element i, y element i + 32:  x' = fma(x, cos, -(y sin))
    // c >= 4: x is element i + 32, y element i: x' = fma(x, cos, y sin)
    const float r = (c < 4) ? __fmaf_rn(x[e], cs_c, -__fmul_rn(y[e], cs_s))
                            : __fmaf_rn(x[e], cs_c, __fmul_rn(y[e], cs_s));
    out[e] = __bfloat162float(__float2bfloat16_rn(r));
  }
}

__device__ __forceinline__ void unpack8(const uint4 w, float (&x)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = bf16lo_to_f32(u[e]);
    x[2 * e + 1] = bf16hi_to_f32(u[e]);
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

__global__ void __launch_bounds__(dec::kWarps * 32)
    ne_attn_decode_split_kernel(const __nv_bfloat16* __restrict__ q,
                                const __nv_bfloat16* __restrict__ kc,
                                const __nv_bfloat16* __restrict__ vc, const int* __restrict__ pos,
                                int H, int Tmax, RopeTable rope, float scale_log2,
                                float* __restrict__ part, int chunk, int n_chunks, int* status) {
  using namespace dec;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int cl = lane & 7;   // 16-byte chunk of the row this lane holds
  const int grp = lane >> 3; // which of the warp's 4 keys per round
  __shared__ float red[kWarps][2 + 64];

  int m_pos = __ldg(pos + b);
  const bool bad = (m_pos < 0 || m_pos >= Tmax);
  if (bad && c == 0 && h == 0 && threadIdx.x == 0 && status) atomicCAS(status, 0, NE_DEV_BAD_SEQLEN);
  const int n_keys = bad ? 0 : m_pos + 1;
  const int k0 = c * chunk + 4 * warp;                        // this warp's first key
  const int k_end = min(c * chunk + chunk, n_keys);

  // q' = R(m) q, the 8 dims of chunk cl (every lane group holds a copy).
  float qr[8];
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(q + (static_cast<long long>(b) * H + h) * 64);
    const uint4 w = __ldg(qrow + cl);
    float x[8], y[8];
    float4 t[4];
    load_pairs(rope.cs + static_cast<long long>(bad ? 0 : m_pos) * 32, cl, t);
    unpack8(w, x);
    unpack8(shfl_xor_u4(w, 4), y);
    rope_chunk(x, y, cl, t, qr);
  }

  float m = -INFINITY, l = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const long long row_stride = static_cast<long long>(H) * 64;  // elements between positions
  const __nv_bfloat16* kb = kc + (static_cast<long long>(b) * Tmax * H + h) * 64;
  const __nv_bfloat16* vb = vc + (static_cast<long long>(b) * Tmax * H + h) * 64;
  // Rounds of 16 keys (4 per warp), in batches of 4 rounds whose loads (K, V
  // and the keys' table rows) are all issued before any of them is used.
  constexpr int kBatch = 4;
  const int rounds = chunk / 16;
  for (int r0 = 0; r0 < rounds; r0 += kBatch) {
    if (k0 + 16 * r0 >= k_end) break;  // warp-uniform: no key of this batch is attended
    uint4 wk[kBatch], wv[kBatch];
    float4 tb[kBatch][4];
    bool live[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int key = k0 + 16 * (r0 + u) + grp;
      live[u] = key < k_end;
      // A key past the end reads row 0 instead, whose value is then ignored:
      // every address formed is inside the cache (read-only loads may run
      // ahead of the condition that guards them).
      const int key_ld = live[u] ? key : 0;
      wk[u] = __ldg(reinterpret_cast<const uint4*>(kb + key_ld * row_stride) + cl);
      wv[u] = __ldg(reinterpret_cast<const uint4*>(vb + key_ld * row_stride) + cl);
      load_pairs(rope.cs + static_cast<long long>(key_ld) * 32, cl, tb[u]);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      float x[8], y[8], kr[8];
      unpack8(wk[u], x);
      unpack8(shfl_xor_u4(wk[u], 4), y);
      rope_chunk(x, y, cl, tb[u], kr);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = __fmaf_rn(qr[e], kr[e], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      dot += __shfl_xor_sync(0xffffffffu, dot, 4);
      if (live[u]) {
        const float sc = dot * scale_log2;
        const float mn = fmaxf(m, sc);
        const float a = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
        const float p = ex2_approx(sc - mn);
        float vv[8];
        unpack8(wv[u], vv);
        l = l * a + p;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __fmaf_rn(p, vv[e], o[e] * a);
        m = mn;
      }
    }
  }
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
  __syncthreads();
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
  float M = -INFINITY;
  for (int c = lane; c < n_chunks; c += 32) M = fmaxf(M, src[c * kPartFloats]);
#pragma unroll
  for (int sh = 16; sh >= 1; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
  float L = 0.f, o0 = 0.f, o1 = 0.f;  // lane owns dims 2*lane, 2*lane + 1
  for (int c = 0; c < n_chunks; ++c) {
    const float* pc = src + c * kPartFloats;
    const float mc = pc[0];
    if (mc == -INFINITY) continue;
    const float a = ex2_approx(mc - M);
    L += pc[1] * a;
    const float2 oc = reinterpret_cast<const float2*>(pc + 4)[lane];
    o0 = __fmaf_rn(oc.x, a, o0);
    o1 = __fmaf_rn(oc.y, a, o1);
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  reinterpret_cast<uint32_t*>(out + bh * 64)[lane] = pack_bf16x2(o0 * inv, o1 * inv);
  if (lane == 0) lse[bh] = (L > 0.f) ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

int decode_chunks(int Tmax) { return (Tmax + dec::kChunkUnit - 1) / dec::kChunkUnit; }

size_t decode_part_bytes(int B, int H, int Tmax) {
  return static_cast<size_t>(B) * H * decode_chunks(Tmax) * dec::kPartFloats * sizeof(float);
}

cudaError_t launch_decode(const __nv_bfloat16* q, const __nv_bfloat16* kc,
                          const __nv_bfloat16* vc, const int* pos, int B, int H, int Tmax,
                          const RopeTable& rope, float scale_log2, float* part,
                          __nv_bfloat16* out, float* lse, int* status, cudaStream_t stream) {
  // 256 keys per CTA measured faster than larger chunks sized to fill the
  // GPU in a few waves (2.5 against 2.0 TB/s at B8 H12 Tmax16384).
  const int chunk = dec::kChunkUnit;
  const int n_chunks = decode_chunks(Tmax);
  dim3 grid(n_chunks, H, B);
  ne_attn_decode_split_kernel<<<grid, dec::kWarps * 32, 0, stream>>>(
      q, kc, vc, pos, H, Tmax, rope, scale_log2, part, chunk, n_chunks, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ne_attn_decode_merge_kernel<<<B * H, 32, 0, stream>>>(part, n_chunks, out, lse);
  return cudaGetLastError();
}

}  // namespace ne
