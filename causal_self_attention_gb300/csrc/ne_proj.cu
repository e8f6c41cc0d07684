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
// 128 x 256 output tiles (128 x 192 for the output projection and dh where
// that makes fewer, fuller rounds of tiles: a 768-wide output in 256-wide
// tiles over 8192 rows is 192 tiles for 152 SMs, the second round a quarter
// full); per tile the K dimension streams through a 4-stage TMA ring of
// 64-column chunks (A 128 x 64, W 256 x 64, 128-byte swizzled).  Two TMEM
// accumulators of 256 (192) columns let the epilogue of one tile overlap the
// MMAs of the next.
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
// block, TMA-loaded into the staging buffer one block ahead, is added;
// kMtpCe -- the tile's 256 columns are one head's logits over a 256-way
// vocabulary: softmax cross-entropy against the row's target, the row's loss
// out, and softmax - onehot (bf16) stored as dlogits; kScale -- the tile
// times 1/n (n: the cross-entropy's target count), bf16; kReduceF32 -- the
// same in fp32, added into the output by bulk tensor reduce-adds (split-K
// partial tiles).
//
// Operand layouts: A and W are K-major by default (A [M, K], W [N, K],
// 64-column chunks); with kAMn / kBMn the operand is read MN-major from a
// [K, M] (or [K, N]) row-major matrix, each 64-row chunk as 64 x 64 boxes
// (8 KiB apart), so that A^T B and A B products need no transposed copies.
// Split-K: a tile list entry is (output tile, K range); its partial result
// is reduced into the output (kReduceF32 only).
//
// Multi-token prediction head (NanoEuler Show HN page, paragraph 2: the MTP
// layers' analytic gradients are checked against double-precision finite
// differences): logits = h . W^T with kMtpCe, then dh = dlogits . W (A
// K-major, W MN-major, kScale) and dW = dlogits^T . h (both MN-major,
// split-K, kReduceF32).
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace gemm {

constexpr int kThreads = 192;
constexpr int kTM = 128, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kTM * kBK * 2;        // 16 KiB
constexpr int kOutBlock = kTM * 64 * 2;       // one 128 x 64 bf16 output block: 16 KiB
constexpr int kBarBytes = 256;
constexpr int kMnBox = 64 * kBK * 2;          // one 64 x 64 box of an MN-major operand: 8 KiB
// Output tiles 128 x kTN: kTN = 256, or 192 where a wave of 128 x 256 tiles
// would leave most SMs idle in its last round (a 768-wide output).
template <int kTN>
struct Tile {
  static_assert(kTN % 64 == 0 && kTN <= 256, "tile width");
  static constexpr int kWBytes = kTN * kBK * 2;  // 32 / 24 KiB
  static constexpr int kStageBytes = kABytes + kWBytes;
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_OUT = OFF_STAGE + kStages * kStageBytes;  // 2 staging buffers
  static constexpr int OFF_BAR = OFF_OUT + 2 * kOutBlock;
  static constexpr int SMEM_BYTES = OFF_BAR + kBarBytes + 1024;  // + slack for alignment
  static_assert(SMEM_BYTES <= 232448, "more shared memory than an sm_103 CTA may have");
};

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


// Entry `t` of the tile list: output tile m fastest (the CTAs working at the
// same time share the weight tile), then n, then the K range.
template <int kTN>
__device__ __forceinline__ void tile_coords(const Params& p, int t, int& m0, int& n0, int& kc0,
                                            int& kc1) {
  const int n_mn = p.n_tiles_m * p.n_tiles_n;
  const int mn = t % n_mn, sp = t / n_mn;
  m0 = (mn % p.n_tiles_m) * kTM;
  n0 = (mn / p.n_tiles_m) * kTN;
  const int k_chunks = (p.K + kBK - 1) / kBK;
  kc0 = sp * p.chunks_per_split;
  kc1 = min(k_chunks, kc0 + p.chunks_per_split);
}

}  // namespace gemm

template <int kEpi, bool kAMn, bool kBMn, int kTN>
__global__ void __launch_bounds__(gemm::kThreads, 1)
    ne_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmO0,   // q' | y | dlogits | dh | dW (fp32)
                   const __grid_constant__ CUtensorMap tmO1,   // k' | residual
                   const __grid_constant__ CUtensorMap tmO2,   // v
                   const gemm::Params p) {
  using namespace gemm;
  constexpr int kStageBytes = Tile<kTN>::kStageBytes;
  constexpr int OFF_STAGE = Tile<kTN>::OFF_STAGE, OFF_OUT = Tile<kTN>::OFF_OUT,
                OFF_BAR = Tile<kTN>::OFF_BAR;
  constexpr int kNB = kTN / 64;  // 64-column output blocks per tile
  constexpr uint32_t kIdesc = make_idesc_bf16(kTM, kTN, kAMn, kBMn);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_tiles = p.n_tiles_m * p.n_tiles_n * p.k_splits;
  const int G = gridDim.x, cta = blockIdx.x;

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
        int m0, n0, kc0, kc1;
        tile_coords<kTN>(p, t, m0, n0, kc0, kc1);
        for (int kb = kc0; kb < kc1; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages &&
              !mbar_wait(&bars[B_EMPTY + s], ((it - kStages) / kStages) & 1, abort_flag, p.status,
                         60)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + OFF_STAGE + s * kStageBytes;
          mbar_arrive_expect_tx(&bars[B_FULL + s], kStageBytes);
          if constexpr (kAMn) {  // A^T chunk: rows kb*64.., columns m0.. of the [K, M] matrix
            tma_load_2d(st, &tmA, &bars[B_FULL + s], m0, kb * kBK);
            tma_load_2d(st + kABytes / 2, &tmA, &bars[B_FULL + s], m0 + 64, kb * kBK);
          } else {
            tma_load_2d(st, &tmA, &bars[B_FULL + s], kb * kBK, m0);
          }
          if constexpr (kBMn) {  // W^T chunk: rows kb*64.., columns n0.. of the [K, N] matrix
#pragma unroll
            for (int i = 0; i < kTN / 64; ++i)
              tma_load_2d(st + kABytes + i * kMnBox, &tmW, &bars[B_FULL + s], n0 + 64 * i,
                          kb * kBK);
          } else {
            tma_load_2d(st + kABytes, &tmW, &bars[B_FULL + s], kb * kBK, n0);
          }
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
    // K-major operand: a K16 step adds 32 bytes; MN-major (64 x 64 boxes 8 KiB
    // apart, 128-byte rows along K): a K16 step adds 16 rows = 2048 bytes.
    const uint64_t dA0 = make_sdesc_sw128(smem_u32(smem + OFF_STAGE), kAMn ? kABytes / 2 : 16, 1024);
    const uint64_t dW0 =
        make_sdesc_sw128(smem_u32(smem + OFF_STAGE + kABytes), kBMn ? kMnBox : 16, 1024);
    constexpr uint64_t kStageD = kStageBytes >> 4;
    constexpr uint64_t kStepA = kAMn ? 128 : 2, kStepW = kBMn ? 128 : 2;
    int it = 0, lt = 0;
    bool ok = true;
    for (int t = cta; ok && t < n_tiles; t += G, ++lt) {
      int m0, n0, kc0, kc1;
      tile_coords<kTN>(p, t, m0, n0, kc0, kc1);
      const int acc = lt & 1;
      if (lt >= 2 &&
          !mbar_wait_warp(&bars[B_ACC_EMPTY + acc], ((lt - 2) >> 1) & 1, abort_flag, p.status, 61)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = kc0; kb < kc1; ++kb, ++it) {
        const int s = it % kStages;
        if (!mbar_wait_warp(&bars[B_FULL + s], (it / kStages) & 1, abort_flag, p.status, 62)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t dA = opaque_u64(dA0) + kStageD * s, dW = opaque_u64(dW0) + kStageD * s;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_ss(tmem + acc * kTN, dA + kStepA * kk, dW + kStepW * kk, kIdesc,
                         (kb > kc0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars[B_EMPTY + s]);
          if (kb == kc1 - 1) umma_commit(&bars[B_ACC_FULL + acc]);
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
      if (kEpi == kQkvRope || kEpi == kResidual) tma_prefetch_desc(&tmO1);
      if (kEpi == kQkvRope) tma_prefetch_desc(&tmO2);
    }
    // Residual block b (over the CTA's tiles x kNB blocks) into staging buffer
    // b & 1: issued by the leader one block ahead.
    auto issue_residual = [&](int b) {
      const int t = cta + (b / kNB) * G;
      if (t >= n_tiles) return;
      int m0, n0, kc0, kc1;
      tile_coords<kTN>(p, t, m0, n0, kc0, kc1);
      mbar_arrive_expect_tx(&bars[B_RES_FULL + (b & 1)], kOutBlock);
      tma_load_2d(stage_out + (b & 1) * kOutBlock, &tmO1, &bars[B_RES_FULL + (b & 1)],
                  n0 + (b % kNB) * 64, m0);
    };
    if (kEpi == kResidual && leader) issue_residual(0);
    // kScale / kReduceF32: the products are the gradients of the mean
    // cross-entropy, 1/n times the sums (n from the cross-entropy kernel,
    // which completed before this grid started).
    float inv_n = 1.f;
    if constexpr (kEpi == kScale || kEpi == kReduceF32) {
      const float cnt = p.acc[1];
      inv_n = cnt > 0.f ? 1.f / cnt : 0.f;
      if (kEpi == kScale && cta == 0 && leader) p.loss[0] = cnt > 0.f ? p.acc[0] / cnt : 0.f;
    }
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;
    int lt = 0, gb = 0;  // tiles, 64-column blocks of this CTA
    for (int t = cta; ok && t < n_tiles; t += G, ++lt) {
      int m0, n0, kc0, kc1;
      tile_coords<kTN>(p, t, m0, n0, kc0, kc1);
      const int acc = lt & 1;
      bool wok = mbar_wait_warp(&bars[B_ACC_FULL + acc], (lt >> 1) & 1, abort_flag, p.status, 63);
      // The token's position (q, k rotation) and its table row, loaded once per tile.
      const int which = (kEpi == kQkvRope) ? n0 / p.C : 0;  // 0 q, 1 k, 2 v
      RopeRow tab;
      if (kEpi == kQkvRope && which < 2) {
        const int row = m0 + r < p.M ? m0 + r : p.M - 1;
        rope_load_row_flat(p.rope, row % p.T, tab);
      }
      // kMtpCe, first pass over the row's 256 logits: max, sum of exponentials
      // (online over the four blocks), the target's logit.
      const int head = (kEpi == kMtpCe) ? n0 / kTN : 0;
      const bool in_rows = m0 + r < p.M;
      int y = -1;
      float lse = 0.f, y_logit = 0.f;
      if constexpr (kEpi == kMtpCe) {
        if (in_rows) y = __ldg(p.targets + static_cast<long long>(m0 + r) * p.heads + head);
        if (wok) {
          tc_fence_after();
          float mx = -INFINITY, se = 0.f;
#pragma unroll 1
          for (int cb = 0; cb < kTN / 64; ++cb) {
            uint32_t v0[32], v1[32];
            tmem_ld_x32(tmem + lane_base + acc * kTN + cb * 64, v0);
            tmem_ld_x32(tmem + lane_base + acc * kTN + cb * 64 + 32, v1);
            tmem_ld_wait(v0);
            tmem_ld_wait(v1);
            float bm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              bm = fmaxf(bm, fmaxf(__uint_as_float(v0[i]), __uint_as_float(v1[i])));
            const float nm = fmaxf(mx, bm);
            float bs = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              bs += ex2_approx((__uint_as_float(v0[i]) - nm) * kLog2e);
              bs += ex2_approx((__uint_as_float(v1[i]) - nm) * kLog2e);
              y_logit = (cb * 64 + i == y) ? __uint_as_float(v0[i]) : y_logit;
              y_logit = (cb * 64 + 32 + i == y) ? __uint_as_float(v1[i]) : y_logit;
            }
            se = se * ex2_approx((mx - nm) * kLog2e) + bs;
            mx = nm;
          }
          lse = mx + logf(se);
        }
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
        if constexpr (kEpi == kReduceF32) {
          // Both staging buffers hold this block as fp32 columns 0-31 and
          // 32-63 ([128][32], 128-byte swizzle); they are free once the
          // previous block's reduce-adds have read them.
          if (leader) bulk_wait_group_read0();
          if (!(ok = named_bar_and(1, 128, ok && wok))) break;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<float4*>(stage_out + h * kOutBlock + sw128_offset(r, c)) =
                  make_float4(a[32 * h + 4 * c] * inv_n, a[32 * h + 4 * c + 1] * inv_n,
                              a[32 * h + 4 * c + 2] * inv_n, a[32 * h + 4 * c + 3] * inv_n);
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (leader) {  // no box starts past the output's last column
            if (n0 + cb * 64 < p.N) tma_reduce_add_2d(&tmO0, stage_out, n0 + cb * 64, m0);
            if (n0 + cb * 64 + 32 < p.N)
              tma_reduce_add_2d(&tmO0, stage_out + kOutBlock, n0 + cb * 64 + 32, m0);
            bulk_commit_group();
          }
          continue;
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
        } else if (kEpi == kMtpCe) {
          // dlogits = softmax - onehot(target); 0 without a target.
#pragma unroll
          for (int i = 0; i < 64; ++i)
            a[i] = y >= 0 ? ex2_approx((a[i] - lse) * kLog2e) - (cb * 64 + i == y ? 1.f : 0.f)
                          : 0.f;
        } else if (kEpi == kScale) {
#pragma unroll
          for (int i = 0; i < 64; ++i) a[i] *= inv_n;
        }
        if (kEpi == kResidual) {
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
        } else {
          // The staging buffer's previous store has read it (the leader waits,
          // all four warps meet; a failed wait above is voted out here).
          if (leader) bulk_wait_group_read1();
          if (!(ok = named_bar_and(1, 128, ok && wok))) break;
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
          } else if (n0 + cb * 64 < p.N) {  // no box starts past the output's last column
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
      if constexpr (kEpi == kMtpCe) {
        // The row's loss (0 without a target); the CTA-wide sums go to acc.
        const bool has = ok && wok && in_rows && y >= 0;
        const float rl = has ? lse - y_logit : 0.f;
        if (ok && wok && in_rows) p.row_loss[static_cast<long long>(m0 + r) * p.heads + head] = rl;
        float sum = rl, cnt = has ? 1.f : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          sum += __shfl_xor_sync(0xffffffffu, sum, o);
          cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        }
        if (lane == 0 && cnt > 0.f) {
          atomicAdd(p.acc, sum);
          atomicAdd(p.acc + 1, cnt);
        }
      }
    }
    if (leader) bulk_wait_group0();  // the stores have completed before the kernel ends
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

namespace {
template <int kEpi, bool kAMn, bool kBMn, int kTN = 256>
cudaError_t launch_gemm_inst(const CUtensorMap& tmA, const CUtensorMap& tmW,
                             const CUtensorMap& tmO0, const CUtensorMap& tmO1,
                             const CUtensorMap& tmO2, const gemm::Params& p, int G,
                             cudaStream_t stream) {
  constexpr int kSmem = gemm::Tile<kTN>::SMEM_BYTES;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(ne_gemm_kernel<kEpi, kAMn, kBMn, kTN>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(ne_gemm_kernel<kEpi, kAMn, kBMn, kTN>, dim3(G), dim3(gemm::kThreads), kSmem,
                    stream, tmA, tmW, tmO0, tmO1, tmO2, p);
}
}  // namespace

// The output tile width for a product of M x N: 192 instead of 256 where it
// takes fewer tile-widths of work on the busiest of G CTAs (rounds of G tiles
// x tile width), for the epilogues built with both (kResidual, kScale).
int gemm_tile_n(int epi, long long M, int N, int G) {
  if ((epi != gemm::kResidual && epi != gemm::kScale) || G <= 0) return 256;
  const long long mt = (M + gemm::kTM - 1) / gemm::kTM;
  auto cost = [&](int tn) { return ((mt * ((N + tn - 1) / tn) + G - 1) / G) * tn; };
  return cost(192) < cost(256) ? 192 : 256;
}

// epi: gemm::Epilogue.  kScale reads A K-major and W MN-major (dlogits . W);
// kReduceF32 reads both MN-major (dlogits^T . h); the others both K-major.
cudaError_t launch_gemm(int epi, const CUtensorMap& tmA, const CUtensorMap& tmW,
                        const CUtensorMap& tmO0, const CUtensorMap& tmO1, const CUtensorMap& tmO2,
                        const gemm::Params& p, cudaStream_t stream) {
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sm_count[dev] &&
      (e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long n_tiles = static_cast<long long>(p.n_tiles_m) * p.n_tiles_n * p.k_splits;
  const int G = static_cast<int>(n_tiles < sm_count[dev] ? n_tiles : sm_count[dev]);
  switch (epi) {
    case gemm::kQkvRope:
      return launch_gemm_inst<gemm::kQkvRope, false, false>(tmA, tmW, tmO0, tmO1, tmO2, p, G, stream);
    case gemm::kResidual:
      if (p.tile_n == 192)
        return launch_gemm_inst<gemm::kResidual, false, false, 192>(tmA, tmW, tmO0, tmO1, tmO2, p,
                                                                    G, stream);
      return launch_gemm_inst<gemm::kResidual, false, false>(tmA, tmW, tmO0, tmO1, tmO2, p, G, stream);
    case gemm::kMtpCe:
      return launch_gemm_inst<gemm::kMtpCe, false, false>(tmA, tmW, tmO0, tmO1, tmO2, p, G, stream);
    case gemm::kScale:
      if (p.tile_n == 192)
        return launch_gemm_inst<gemm::kScale, false, true, 192>(tmA, tmW, tmO0, tmO1, tmO2, p, G,
                                                                stream);
      return launch_gemm_inst<gemm::kScale, false, true>(tmA, tmW, tmO0, tmO1, tmO2, p, G, stream);
    case gemm::kReduceF32:
      return launch_gemm_inst<gemm::kReduceF32, true, true>(tmA, tmW, tmO0, tmO1, tmO2, p, G, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ne
