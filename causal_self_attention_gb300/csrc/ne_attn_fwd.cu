// ne_attn_fwd.cu -- forward causal self-attention with fused RoPE on sm_103a.
//
// One CTA computes one 128-row query tile of one (sequence, head):
//   O_m = sum_{n<=m} softmax_n(scale * q'_m . k'_n) v_n,  LSE_m = log sum exp(...)
// with q' = R(m) q, k' = R(n) k (RoPE), the scores never leaving the SM
// (tiled online softmax, as in the hand-written FlashAttention of the
// NanoEuler Show HN page, paragraph 2; causality as in "Tiny Hackable CUDA",
// section 3).
//
// Warp roles (320 threads):
//   warps 0-3  rotate: RoPE on the Q tile once and on every K tile in smem
//   warps 4-7  softmax: thread t owns query row t (TMEM lane t); online
//              softmax with a lazily moved reference max, P to smem, O
//              rescale in TMEM, epilogue (O / l, LSE)
//   warp 8     MMA: allocates TMEM; lane 0 issues S = Q K^T and O += P V
//   warp 9     TMA: lane 0 loads Q once and K/V tiles into a 2-stage ring
// TMEM: S double buffer (2 x 128 fp32 columns) + O (64 columns).
// Key tiles entirely above the diagonal are never loaded or computed.
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace fwd {

constexpr int kThreads = 320;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + kTileBytes;        // 2 stages
constexpr int OFF_V = OFF_K + 2 * kTileBytes;    // 2 stages
constexpr int OFF_P = OFF_V + 2 * kTileBytes;    // 2 buffers x (2 x 16 KiB)
constexpr int OFF_BAR = OFF_P + 4 * kTileBytes;  // barriers + scalars
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + slack for 1024-byte alignment

enum Bar {
  B_Q_FULL = 0,
  B_Q_ROT,
  B_KV_FULL,   // 2
  B_K_ROT = B_KV_FULL + 2,
  B_KV_EMPTY = B_K_ROT + 2,
  B_S_FULL = B_KV_EMPTY + 2,
  B_S_FREE = B_S_FULL + 2,
  B_P_FULL = B_S_FREE + 2,
  B_PV_DONE = B_P_FULL + 2,
  B_MMA_DONE = B_PV_DONE + 2,
  B_COUNT
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;  // O at columns 256..319

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);  // Q K^T
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, false, true);    // P V (V MN-major)

}  // namespace fwd

__global__ void __launch_bounds__(fwd::kThreads, 1)
    ne_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);

  // ---- which tile: longest (last) query tiles first --------------------------
  const int H = p.pb.H;
  const int seq = blockIdx.x / H;
  const int h = blockIdx.x % H;
  const int qt = gridDim.y - 1 - blockIdx.y;
  int start, len;
  if (!seq_bounds(p.pb, seq, start, len, (qt == 0 && threadIdx.x == 0) ? p.status : nullptr))
    return;
  if (qt * kBM >= len) return;  // whole CTA: this sequence has no such tile
  const int n_kv = qt + 1;       // causal: key tiles 0..qt
  const int row0 = start + qt * kBM;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_Q_ROT], 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_KV_FULL + s], 1);
      mbar_init(&bars[B_K_ROT + s], 128);
      mbar_init(&bars[B_KV_EMPTY + s], 1);
      mbar_init(&bars[B_S_FULL + s], 1);
      mbar_init(&bars[B_S_FREE + s], 128);
      mbar_init(&bars[B_P_FULL + s], 128);
      mbar_init(&bars[B_PV_DONE + s], 1);
    }
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sP = smem + OFF_P;

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars[B_Q_FULL], kTileBytes);
      tma_load_3d(sQ, &tmQ, &bars[B_Q_FULL], 0, h, row0);
      int last_issued[2] = {-1, -1};
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(&bars[B_KV_EMPTY + s], ((j - 2) >> 1) & 1, abort_flag, p.status, 1))
          break;
        mbar_arrive_expect_tx(&bars[B_KV_FULL + s], 2 * kTileBytes);
        tma_load_3d(sK + s * kTileBytes, &tmK, &bars[B_KV_FULL + s], 0, h, start + j * kBN);
        tma_load_3d(sV + s * kTileBytes, &tmV, &bars[B_KV_FULL + s], 0, h, start + j * kBN);
        last_issued[s] = j;
      }
      if (*abort_flag) {
        // Let the copies still in flight land before the CTA exits.
        mbar_wait(&bars[B_Q_FULL], 0, abort_flag, nullptr, 0);
        for (int s = 0; s < 2; ++s)
          if (last_issued[s] >= 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[B_KV_FULL + s], (last_issued[s] >> 1) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t aQ = smem_u32(sQ);
      bool ok = mbar_wait(&bars[B_Q_ROT], 0, abort_flag, p.status, 2);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj & 1;
        if (!mbar_wait(&bars[B_P_FULL + s], (jj >> 1) & 1, abort_flag, p.status, 3)) return false;
        tc_fence_after();
        const uint32_t aP = smem_u32(sP + s * 2 * kTileBytes);
        const uint32_t aV = smem_u32(sV + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // K = 128 keys in steps of 16
          const uint64_t da =
              make_sdesc_sw128(aP + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t db = make_sdesc_sw128(aV + kk * 2048, 16 * 1024, 1024);
          umma_bf16_ss(tmem + kColO, da, db, kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_PV_DONE + s]);
        umma_commit(&bars[B_KV_EMPTY + s]);
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&bars[B_K_ROT + s], (j >> 1) & 1, abort_flag, p.status, 4)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(&bars[B_S_FREE + s], ((j - 2) >> 1) & 1, abort_flag, p.status, 5)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // K = 64 head dims in steps of 16
          const uint64_t da = make_sdesc_sw128(aQ + kk * 32, 16, 1024);
          const uint64_t db = make_sdesc_sw128(aK + kk * 32, 16, 1024);
          umma_bf16_ss(tmem + kColS + s * 128, da, db, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[B_S_FULL + s]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_kv - 1);
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit(&bars[B_MMA_DONE]);
      const long long t0 = clock64();
      while (!mbar_try_wait(&bars[B_MMA_DONE], 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ RoPE warps
    const int r = threadIdx.x;  // 0..127: tile row
    if (mbar_wait(&bars[B_Q_FULL], 0, abort_flag, p.status, 6)) {
      rope_rotate_row(sQ, r, qt * kBM + r, p.rope);
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_Q_ROT]);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&bars[B_KV_FULL + s], (j >> 1) & 1, abort_flag, p.status, 7)) break;
        rope_rotate_row(sK + s * kTileBytes, r, j * kBN + r, p.rope);
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_K_ROT + s]);
      }
    }
  } else {
    // --------------------------------------------------------- softmax warps
    const int wq = warp - 4;          // TMEM lane quarter
    const int r = wq * 32 + lane;     // query row in tile
    const int qpos = qt * kBM + r;    // position in sequence
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    float m_ref = -INFINITY;  // reference max (log2 units) the P values are taken against
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      if (!mbar_wait_warp(&bars[B_S_FULL + s], (j >> 1) & 1, abort_flag, p.status, 8)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      const uint32_t tS = tmem + lane_base + kColS + s * 128;
      tmem_ld_x32(tS + 0, sr + 0);
      tmem_ld_x32(tS + 32, sr + 32);
      tmem_ld_x32(tS + 64, sr + 64);
      tmem_ld_x32(tS + 96, sr + 96);
      tmem_ld_wait(sr + 0);
      tmem_ld_wait(sr + 32);
      tmem_ld_wait(sr + 64);
      tmem_ld_wait(sr + 96);
      tc_fence_before();
      mbar_arrive(&bars[B_S_FREE + s]);

      float x[128];
      float mx = -INFINITY;
      const bool diag = (j == qt);
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        float v = __uint_as_float(sr[c]) * p.scale_log2;
        if (diag && c > r) v = -INFINITY;  // key j*128+c after query qt*128+r
        x[c] = v;
        mx = fmaxf(mx, v);
      }
      // Move the reference max only when the row max grows by more than 2^8;
      // otherwise keep it (exact: O and l share the same reference).
      const bool need = (mx > m_ref + 8.0f);
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mx);
        m_ref = mx;
      }
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        x[c] = ex2_approx(x[c] - m_ref);
        rs += x[c];
      }
      l_sum = l_sum * alpha + rs;

      const bool warp_rescale = __any_sync(0xffffffffu, need && j > 0);
      if (warp_rescale) {
        // O must be stable: wait for the P V of the previous tile.
        if (!mbar_wait_warp(&bars[B_PV_DONE + ((j - 1) & 1)], ((j - 1) >> 1) & 1, abort_flag,
                            p.status, 9)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t o[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          tmem_ld_x32(tO + half * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_x32(tO + half * 32, o);
        }
        tmem_st_wait();
      } else if (j >= 2) {
        // The P buffer about to be written was read by the P V of tile j-2.
        if (!mbar_wait_warp(&bars[B_PV_DONE + s], ((j - 2) >> 1) & 1, abort_flag, p.status, 10)) {
          ok = false;
          break;
        }
      }
      uint8_t* pbuf = sP + s * 2 * kTileBytes;
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        const int c0 = c16 * 8;
        uint4 w;
        w.x = pack_bf16x2(x[c0 + 0], x[c0 + 1]);
        w.y = pack_bf16x2(x[c0 + 2], x[c0 + 3]);
        w.z = pack_bf16x2(x[c0 + 4], x[c0 + 5]);
        w.w = pack_bf16x2(x[c0 + 6], x[c0 + 7]);
        *reinterpret_cast<uint4*>(pbuf + (c16 >> 3) * kTileBytes + sw128_offset(r, c16 & 7)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL + s]);
    }
    // ---- epilogue: O / l and LSE for rows inside the sequence -------------
    if (ok && mbar_wait_warp(&bars[B_PV_DONE + ((n_kv - 1) & 1)], ((n_kv - 1) >> 1) & 1,
                             abort_flag, p.status, 11)) {
      tc_fence_after();
      uint32_t o[64];
      tmem_ld_x32(tO, o);
      tmem_ld_x32(tO + 32, o + 32);
      tmem_ld_wait(o);
      tmem_ld_wait(o + 32);
      if (qpos < len) {
        const float inv_l = 1.f / l_sum;
        const long long orow = (static_cast<long long>(row0 + r) * H + h) * kHD;
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            dst[c] = make_float4(__uint_as_float(o[4 * c + 0]) * inv_l,
                                 __uint_as_float(o[4 * c + 1]) * inv_l,
                                 __uint_as_float(o[4 * c + 2]) * inv_l,
                                 __uint_as_float(o[4 * c + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * c + 0]) * inv_l, __uint_as_float(o[8 * c + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * c + 2]) * inv_l, __uint_as_float(o[8 * c + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * c + 4]) * inv_l, __uint_as_float(o[8 * c + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * c + 6]) * inv_l, __uint_as_float(o[8 * c + 7]) * inv_l);
            dst[c] = w;
          }
        }
        // LSE in natural-log units: (m_ref + log2 l) * ln 2.
        p.lse[lse_index(p.pb, h, seq, start, qpos)] = (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const FwdParams& p, int n_qtiles, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_attn_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fwd::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(p.pb.nseq * p.pb.H, n_qtiles);
  ne_attn_fwd_kernel<<<grid, fwd::kThreads, fwd::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace ne
