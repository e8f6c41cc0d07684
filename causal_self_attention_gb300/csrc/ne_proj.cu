// ne_proj.cu -- the projections around the attention, on sm_103a: RMSNorm,
// then the QKV projection with RoPE applied in the GEMM's epilogue (so the
// attention can take q' = R(m) q and k' = R(n) k as they are), and the output
// projection with the residual added in the epilogue.  (NanoEuler Show HN
// page, paragraph 2: the CUDA engine has RMSNorm and RoPE kernels and computes
// the matrix products of the layer; "Tiny Hackable CUDA", section 3: the
// projections are computed, RoPE is applied to them, and the attention is
// wrapped in a residual connection.)
//
// GEMM: Y[M, N] = A[M, K] . W[N, K]^T, bf16 operands, fp32 accumulation,
// weights in the [out, in] layout.  Persistent CTAs (one per SM) walk the
// 128 x 256 output tiles; per tile the K dimension streams through a 4-stage
// TMA ring of 64-column chunks (A 128 x 64, W 256 x 64, 128-byte swizzled).
// Two TMEM accumulators of 256 columns let the epilogue of one tile overlap
// the MMAs of the next.
//   warp 0      TMA: lane 0 loads the A and W chunks
//   warp 1      MMA: allocates TMEM; its elected lane issues the tcgen05 MMAs
//               (M 128, N 256, K 16)
//   warps 2-5   epilogue: thread t owns output row t of the tile (TMEM lane
//               t); per 64-column block it loads the accumulator row, applies
//               the epilogue, writes the bf16 row into a swizzled staging
//               buffer, and one thread stores the block with TMA (two staging
//               buffers, so a block's store overlaps the next block)
// Epilogues: kQkvRope -- the tile lies in q, k or v (C is a multiple of 256);
// q and k columns are rotated per head of 64 at the token's position
// (row mod T) in fp32 before the bf16 rounding; kResidual -- the residual
// block, TMA-loaded into the staging buffer one block ahead, is added.
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace gemm {

constexpr int kThreads = 192;
constexpr int kTM = 128, kTN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kTM * kBK * 2;        // 16 KiB
constexpr int kWBytes = kTN * kBK * 2;        // 32 KiB
constexpr int kStageBytes = kABytes + kWBytes;
constexpr int kOutBlock = kTM * 64 * 2;       // one 128 x 64 bf16 output block: 16 KiB
constexpr int OFF_STAGE = 0;
constexpr int OFF_OUT = OFF_STAGE + kStages * kStageBytes;  // 2 staging buffers
constexpr int OFF_BAR = OFF_OUT + 2 * kOutBlock;
constexpr int kBarBytes = 256;
constexpr int SMEM_BYTES = OFF_BAR + kBarBytes + 1024;  // + slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "more shared memory than an sm_103 CTA may have");

enum Bar {
  B_FULL = 0,                  // kStages
  B_EMPTY = B_FULL + kStages,  // kStages
  B_ACC_FULL = B_EMPTY + kStages,  // 2
  B_ACC_EMPTY = B_ACC_FULL + 2,    // 2
  B_RES_FULL = B_ACC_EMPTY + 2,    // 2 (per staging buffer)
  B_MMA_DONE = B_RES_FULL + 2,
  B_COUNT
};
static_assert(8 * B_COUNT + 8 <= kBarBytes, "barrier region overflow");

constexpr uint32_t kIdesc = make_idesc_bf16(kTM, kTN, false, false);  // A, W both K-major

enum Epilogue { kQkvRope = 0, kResidual = 1 };

struct Params {
  int M, N, K;
  int n_tiles_m, n_tiles_n;
  int C;          // kQkvRope: width of each of q, k, v (N = 3C)
  int T;          // kQkvRope: tokens per sequence (position = row mod T)
  RopeTable rope;
  int* status;
};

// Tile `t` of the output: m fastest, so the CTAs working at the same time
// share the weight tile (3.5 MB of weights stay in L2 either way).
__device__ __forceinline__ void tile_coords(const Params& p, int t, int& m0, int& n0) {
  m0 = (t % p.n_tiles_m) * kTM;
  n0 = (t / p.n_tiles_m) * kTN;
}

}  // namespace gemm

template <int kEpi>
__global__ void __launch_bounds__(gemm::kThreads, 1)
    ne_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmO0,   // q' | y
                   const __grid_constant__ CUtensorMap tmO1,   // k' | residual
                   const __grid_constant__ CUtensorMap tmO2,   // v
                   const gemm::Params p) {
  using namespace gemm;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_tiles = p.n_tiles_m * p.n_tiles_n;
  const int G = gridDim.x, cta = blockIdx.x;
  const int k_chunks = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_FULL + s], 1);
      mbar_init(&bars[B_EMPTY + s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars[B_ACC_FULL + a], 1);
      mbar_init(&bars[B_ACC_EMPTY + a], 128);
      mbar_init(&bars[B_RES_FULL + a], 1);
    }
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the kernels that wrote A (and anything before) have completed
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmW);
      int it = 0;  // chunks loaded over all tiles
      int last[kStages] = {-1, -1, -1, -1};
      bool ok = true;
      for (int t = cta; ok && t < n_tiles; t += G) {
        int m0, n0;
        tile_coords(p, t, m0, n0);
        for (int kb = 0; kb < k_chunks; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages &&
              !mbar_wait(&bars[B_EMPTY + s], ((it - kStages) / kStages) & 1, abort_flag, p.status,
                         60)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + OFF_STAGE + s * kStageBytes;
          mbar_arrive_expect_tx(&bars[B_FULL + s], kStageBytes);
          tma_load_2d(st, &tmA, &bars[B_FULL + s], kb * kBK, m0);
          tma_load_2d(st + kABytes, &tmW, &bars[B_FULL + s], kb * kBK, n0);
          last[s] = it;
        }
      }
      if (!ok || *abort_flag)  // copies in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (last[s] >= 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[B_FULL + s], (last[s] / kStages) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMAs
    const uint64_t d0 = make_sdesc_sw128(smem_u32(smem + OFF_STAGE), 16, 1024);
    constexpr uint64_t kStageD = kStageBytes >> 4, kAD = kABytes >> 4;
    int it = 0, lt = 0;
    bool ok = true;
    for (int t = cta; ok && t < n_tiles; t += G, ++lt) {
      const int acc = lt & 1;
      if (lt >= 2 &&
          !mbar_wait_warp(&bars[B_ACC_EMPTY + acc], ((lt - 2) >> 1) & 1, abort_flag, p.status, 61)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < k_chunks; ++kb, ++it) {
        const int s = it % kStages;
        if (!mbar_wait_warp(&bars[B_FULL + s], (it / kStages) & 1, abort_flag, p.status, 62)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dA = opaque_u64(d0) + kStageD * s, dW = dA + kAD;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // 16 elements = 32 bytes per step
            umma_bf16_ss(tmem + acc * kTN, dA + 2 * kk, dW + 2 * kk, kIdesc,
                         (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars[B_EMPTY + s]);
          if (kb == k_chunks - 1) umma_commit(&bars[B_ACC_FULL + acc]);
        }
        __syncwarp();
      }
    }
    if (elect_one()) umma_commit(&bars[B_MMA_DONE]);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(&bars[B_MMA_DONE], 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const bool leader = (warp == 2 && lane == 0);
    uint8_t* stage_out = smem + OFF_OUT;
    if (leader) {
      tma_prefetch_desc(&tmO0);
      tma_prefetch_desc(&tmO1);
      if (kEpi == kQkvRope) tma_prefetch_desc(&tmO2);
    }
    // Residual block b (over the CTA's tiles x 4 blocks) into staging buffer
    // b & 1: issued by the leader one block ahead.
    auto issue_residual = [&](int b) {
      const int t = cta + (b >> 2) * G;
      if (t >= n_tiles) return;
      int m0, n0;
      tile_coords(p, t, m0, n0);
      mbar_arrive_expect_tx(&bars[B_RES_FULL + (b & 1)], kOutBlock);
      tma_load_2d(stage_out + (b & 1) * kOutBlock, &tmO1, &bars[B_RES_FULL + (b & 1)],
                  n0 + (b & 3) * 64, m0);
    };
    if (kEpi == kResidual && leader) issue_residual(0);
    bool ok = true;
    int lt = 0, gb = 0;  // tiles, 64-column blocks of this CTA
    for (int t = cta; ok && t < n_tiles; t += G, ++lt) {
      int m0, n0;
      tile_coords(p, t, m0, n0);
      const int acc = lt & 1;
      bool wok = mbar_wait_warp(&bars[B_ACC_FULL + acc], (lt >> 1) & 1, abort_flag, p.status, 63);
      // The token's position (q, k rotation) and its table row, loaded once per tile.
      const int which = (kEpi == kQkvRope) ? n0 / p.C : 0;  // 0 q, 1 k, 2 v
      RopeRow tab;
      if (kEpi == kQkvRope && which < 2) {
        const int row = m0 + r < p.M ? m0 + r : p.M - 1;
        rope_load_row_flat(p.rope, row % p.T, tab);
      }
      tc_fence_after();
      for (int cb = 0; cb < kTN / 64; ++cb, ++gb) {
        const int sb = gb & 1;
        uint8_t* buf = stage_out + sb * kOutBlock;
        float a[64];
        if (wok) {
          uint32_t v0[32], v1[32];
          tmem_ld_x32(tmem + lane_base + acc * kTN + cb * 64, v0);
          tmem_ld_x32(tmem + lane_base + acc * kTN + cb * 64 + 32, v1);
          tmem_ld_wait(v0);
          tmem_ld_wait(v1);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = __uint_as_float(v0[i]);
            a[32 + i] = __uint_as_float(v1[i]);
          }
        }
        if (cb == kTN / 64 - 1 && wok) {  // the whole accumulator row has been read
          tc_fence_before();
          mbar_arrive(&bars[B_ACC_EMPTY + acc]);
        }
        if (kEpi == kQkvRope) {
          if (which < 2) {
            // RoPE, rotate-half within the head: element i pairs with i + 32,
            // turned by the angle of frequency i at this row's position; in
            // fp32, the table values being the fp32 roundings of the double
            // cos / sin.
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float4 cs = tab.t[i >> 1];  // (cos_i, sin_i, cos_{i+1}, sin_{i+1})
              const float x0 = a[i], y0 = a[i + 32], x1 = a[i + 1], y1 = a[i + 33];
              a[i] = __fmaf_rn(x0, cs.x, -__fmul_rn(y0, cs.y));
              a[i + 32] = __fmaf_rn(y0, cs.x, __fmul_rn(x0, cs.y));
              a[i + 1] = __fmaf_rn(x1, cs.z, -__fmul_rn(y1, cs.w));
              a[i + 33] = __fmaf_rn(y1, cs.z, __fmul_rn(x1, cs.w));
            }
          }
          // The staging buffer's previous store has read it (the leader waits,
          // all four warps meet; a failed wait above is voted out here).
          if (leader) bulk_wait_group_read1();
          if (!(ok = named_bar_and(1, 128, ok && wok))) break;
        } else {
          // The residual block was loaded into this buffer one block ahead.
          wok = wok && mbar_wait_warp(&bars[B_RES_FULL + sb], (gb >> 1) & 1, abort_flag,
                                      p.status, 64);
          if (!(ok = named_bar_and(1, 128, ok && wok))) break;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 rv = *reinterpret_cast<const uint4*>(buf + sw128_offset(r, c));
            a[8 * c + 0] += bf16lo_to_f32(rv.x);
            a[8 * c + 1] += bf16hi_to_f32(rv.x);
            a[8 * c + 2] += bf16lo_to_f32(rv.y);
            a[8 * c + 3] += bf16hi_to_f32(rv.y);
            a[8 * c + 4] += bf16lo_to_f32(rv.z);
            a[8 * c + 5] += bf16hi_to_f32(rv.z);
            a[8 * c + 6] += bf16lo_to_f32(rv.w);
            a[8 * c + 7] += bf16hi_to_f32(rv.w);
          }
        }
        // Row r of the block, bf16, into the swizzled staging buffer.
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(buf + sw128_offset(r, c)) =
              make_uint4(pack_bf16x2(a[8 * c + 0], a[8 * c + 1]), pack_bf16x2(a[8 * c + 2], a[8 * c + 3]),
                         pack_bf16x2(a[8 * c + 4], a[8 * c + 5]), pack_bf16x2(a[8 * c + 6], a[8 * c + 7]));
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          if (kEpi == kQkvRope) {
            const CUtensorMap* out = which == 0 ? &tmO0 : (which == 1 ? &tmO1 : &tmO2);
            tma_store_2d(out, buf, n0 - which * p.C + cb * 64, m0);
          } else {
            tma_store_2d(&tmO0, buf, n0 + cb * 64, m0);
          }
          bulk_commit_group();
          if (kEpi == kResidual) {
            // The other buffer's store (the previous block) has read it: load
            // the residual of the next block there.
            bulk_wait_group_read1();
            issue_residual(gb + 1);
          }
        }
      }
    }
    if (leader) bulk_wait_group0();  // the stores have completed before the kernel ends
    if (kEpi == kResidual && leader) {
      // A residual load issued for a block past the CTA's last tile is never
      // issued (issue_residual skips it); nothing else can be in flight.
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// RMSNorm: one warp per row of C (a multiple of 8): xn = bf16(x * rstd * g),
// rstd = 1 / sqrt(mean(x^2) + eps) accumulated in fp32 (and written out when
// asked, for the backward).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    ne_rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ g,
                      __nv_bfloat16* __restrict__ xn, float* __restrict__ rstd, int M, int C,
                      float eps) {
  pdl_wait();
  const int row = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row < M) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(row) * C);
    float ss = 0.f;
    for (int c = lane; c < C / 8; c += 32) {
      const uint4 w = __ldg(xr + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float lo = bf16lo_to_f32(ws[u]), hi = bf16hi_to_f32(ws[u]);
        ss = __fmaf_rn(lo, lo, ss);
        ss = __fmaf_rn(hi, hi, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.f / sqrtf(ss / static_cast<float>(C) + eps);
    if (rstd && lane == 0) rstd[row] = inv;
    uint4* outr = reinterpret_cast<uint4*>(xn + static_cast<long long>(row) * C);
    const uint4* gr = reinterpret_cast<const uint4*>(g);
    for (int c = lane; c < C / 8; c += 32) {
      const uint4 w = __ldg(xr + c), gw = __ldg(gr + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w}, gs[4] = {gw.x, gw.y, gw.z, gw.w};
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        o[u] = pack_bf16x2(bf16lo_to_f32(ws[u]) * inv * bf16lo_to_f32(gs[u]),
                           bf16hi_to_f32(ws[u]) * inv * bf16hi_to_f32(gs[u]));
      outr[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  pdl_launch_dependents();
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* xn,
                           float* rstd, int M, int C, float eps, cudaStream_t stream) {
  return launch_pdl(ne_rmsnorm_kernel, dim3((M + 7) / 8), dim3(256), 0, stream, x, g, xn, rstd, M,
                    C, eps);
}

cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const CUtensorMap& tmO0, const CUtensorMap& tmO1, const CUtensorMap& tmO2,
                        const gemm::Params& p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_gemm_kernel<gemm::kQkvRope>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gemm::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ne_gemm_kernel<gemm::kResidual>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, gemm::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sm_count[dev] &&
      (e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int n_tiles = p.n_tiles_m * p.n_tiles_n;
  const int G = n_tiles < sm_count[dev] ? n_tiles : sm_count[dev];
  if (epi == gemm::kQkvRope)
    return launch_pdl(ne_gemm_kernel<gemm::kQkvRope>, dim3(G), dim3(gemm::kThreads),
                      gemm::SMEM_BYTES, stream, tmA, tmW, tmO0, tmO1, tmO2, p);
  return launch_pdl(ne_gemm_kernel<gemm::kResidual>, dim3(G), dim3(gemm::kThreads),
                    gemm::SMEM_BYTES, stream, tmA, tmW, tmO0, tmO1, tmO2, p);
}

}  // namespace ne
