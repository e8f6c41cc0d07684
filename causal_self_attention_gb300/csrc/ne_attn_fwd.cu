// ne_attn_fwd.cu -- forward causal self-attention with fused RoPE on sm_103a.
//
// One CTA computes two consecutive 128-row query tiles (A: rows 256p..256p+127,
// B: rows 256p+128..256p+255) of one (sequence, head):
//   O_m = sum_{n<=m} softmax_n(scale * q'_m . k'_n) v_n,  LSE_m = log sum exp(...)
// with q' = R(m) q, k' = R(n) k (RoPE), the scores never leaving the SM
// (tiled online softmax, as in the hand-written FlashAttention of the
// NanoEuler Show HN page, paragraph 2; causality as in "Tiny Hackable CUDA",
// section 3).  Both tiles share every rotated K/V tile, and while one tile's
// softmax runs the tensor core works on the other tile's MMAs.
//
// Warp roles (512 threads, registers re-split per warpgroup with setmaxnreg):
//   warps 0-3   softmax A: thread t owns row t of tile A (TMEM lane t), 168 regs
//   warps 4-7   softmax B: same for tile B
//   warps 8-11  rotate: RoPE on Q_A, Q_B once and on every K tile in smem, 112
//   warp 12     MMA: allocates TMEM; one elected lane issues S_X = Q_X K^T, O_X += P_X V
//   warp 13     TMA: lane 0 loads Q_A, Q_B once and the K ring (5 stages)
//   warp 14     TMA: lane 0 loads the V ring (5 stages); warps 12-15 run at
//               64 regs
// TMEM columns: S_A 0-127, S_B 128-255, O_A 256-319, O_B 320-383,
// P_A 384-447, P_B 448-511 (bf16 pairs: P is the TMEM A operand of P V).
// A softmax thread loads its whole S row with one TMEM round trip and frees
// S_X at once, so the next S_X = Q_X K^T overlaps the exponentials; the
// reference max moves only when the row max grows by more than 2^8 (exact: O
// and l keep a common reference).
// Key tiles entirely above the diagonal are never loaded or computed.
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace fwd {

constexpr int kThreads = 512;
// Registers per thread of each warpgroup after setmaxnreg (launch: 128).
constexpr uint32_t kRegsSoftmax = 168, kRegsRotate = 112, kRegsMma = 64;
static_assert(valid_reg_split(kRegsSoftmax, kRegsRotate, kRegsMma), "register split");
constexpr int kStages = 5;                            // K ring and V ring
constexpr int OFF_Q = 0;                              // Q_A, Q_B
constexpr int OFF_K = OFF_Q + 2 * kTileBytes;         // kStages
constexpr int OFF_V = OFF_K + kStages * kTileBytes;   // kStages
constexpr int OFF_BAR = OFF_V + kStages * kTileBytes;
constexpr int kBarBytes = 512;  // mbarriers, TMEM address, abort flag
constexpr int SMEM_BYTES = OFF_BAR + kBarBytes + 1024;  // + slack for 1024-byte alignment

enum Bar {
  B_Q_FULL = 0,
  B_Q_ROT,
  B_K_FULL,                           // kStages
  B_K_ROT = B_K_FULL + kStages,       // kStages
  B_K_EMPTY = B_K_ROT + kStages,      // kStages
  B_V_FULL = B_K_EMPTY + kStages,     // kStages
  B_V_EMPTY = B_V_FULL + kStages,     // kStages
  B_S_FULL = B_V_EMPTY + kStages,     // per tile X
  B_S_FREE = B_S_FULL + 2,
  B_P_FULL = B_S_FREE + 2,
  B_PV_DONE = B_P_FULL + 2,
  B_O_FINAL = B_PV_DONE + 2,         // once per tile: its last P V completed
  B_MMA_DONE = B_O_FINAL + 2,
  B_COUNT
};
static_assert(8 * B_COUNT + 8 <= kBarBytes, "barrier region overflow");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_X at 128 * X
constexpr uint32_t kColO = 256;  // O_X at 256 + 64 * X
constexpr uint32_t kColP = 384;  // P_X at 384 + 64 * X

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

  // ---- which block of 256 query rows: longest (last) blocks first ----------
  const int H = p.pb.H;
  const int seq = blockIdx.x / H;
  const int h = blockIdx.x % H;
  const int blk = gridDim.y - 1 - blockIdx.y;
  int start, len;
  if (!seq_bounds(p.pb, seq, start, len, (blk == 0 && threadIdx.x == 0) ? p.status : nullptr))
    return;
  const int rowA = 2 * blk * kBM;  // first row of tile A in the sequence
  if (rowA >= len) return;         // whole CTA: this sequence has no such block
  const bool hasB = rowA + kBM < len;
  const int nkvA = 2 * blk + 1;    // causal: key tiles 0..2blk for A, 0..2blk+1 for B
  const int nkvB = hasB ? 2 * blk + 2 : 0;
  const int nkv = hasB ? nkvB : nkvA;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q_FULL], 1);
    mbar_init(&bars[B_Q_ROT], 128);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[B_K_FULL + s], 1);
      mbar_init(&bars[B_K_ROT + s], 128);
      mbar_init(&bars[B_K_EMPTY + s], 1);
      mbar_init(&bars[B_V_FULL + s], 1);
      mbar_init(&bars[B_V_EMPTY + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[B_S_FULL + x], 1);
      mbar_init(&bars[B_S_FREE + x], 128);
      mbar_init(&bars[B_P_FULL + x], 128);
      mbar_init(&bars[B_PV_DONE + x], 1);
      mbar_init(&bars[B_O_FINAL + x], 1);
    }
    mbar_init(&bars[B_MMA_DONE], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 12) {
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

  if (warp == 13 || warp == 14) {
    // ------------------------------------ TMA producers: warp 13 K, warp 14 V
    regs_decrease<kRegsMma>();
    if (lane == 0) {
      const bool isK = (warp == 13);
      const CUtensorMap* tm = isK ? &tmK : &tmV;
      uint8_t* ring = isK ? sK : sV;
      uint64_t* full = &bars[isK ? B_K_FULL : B_V_FULL];
      uint64_t* empty = &bars[isK ? B_K_EMPTY : B_V_EMPTY];
      tma_prefetch_desc(tm);
      if (isK) {
        tma_prefetch_desc(&tmQ);
        mbar_arrive_expect_tx(&bars[B_Q_FULL], 2 * kTileBytes);
        tma_load_3d(sQ, &tmQ, &bars[B_Q_FULL], 0, h, start + rowA);
        tma_load_3d(sQ + kTileBytes, &tmQ, &bars[B_Q_FULL], 0, h, start + rowA + kBM);
      }
      int last_issued[kStages];
      for (int s = 0; s < kStages; ++s) last_issued[s] = -1;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            !mbar_wait(&empty[s], ((j - kStages) / kStages) & 1, abort_flag, p.status, isK ? 1 : 12))
          break;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        tma_load_3d(ring + s * kTileBytes, tm, &full[s], 0, h, start + j * kBN);
        last_issued[s] = j;
      }
      if (*abort_flag) {
        // Let the copies still in flight land before the CTA exits.
        if (isK) mbar_wait(&bars[B_Q_FULL], 0, abort_flag, nullptr, 0);
        for (int s = 0; s < kStages; ++s)
          if (last_issued[s] >= 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&full[s], (last_issued[s] / kStages) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
      }
    }
  } else if (warp == 12) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and waits; the elected lane issues each
    // group of MMAs together with the commit that tracks it.  Shared-memory
    // descriptors are built once: a K step, a tile or a ring stage only adds a
    // constant to the start-address field (16-byte units).
    regs_decrease<kRegsMma>();
    constexpr uint64_t kTileD = kTileBytes >> 4;
    const uint64_t dQ0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);          // Q K-major
    const uint64_t dK0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);          // K K-major
    const uint64_t dV0 = make_sdesc_sw128(smem_u32(sV), kTileBytes, 1024);  // V MN-major
    bool ok = mbar_wait_warp(&bars[B_Q_ROT], 0, abort_flag, p.status, 2);
    for (int j = 0; ok && j <= nkv; ++j) {
      if (j < nkv) {
        const int s = j % kStages;
        if (!mbar_wait_warp(&bars[B_K_ROT + s], (j / kStages) & 1, abort_flag, p.status, 3)) {
          ok = false;
          break;
        }
        const uint64_t dK = dK0 + kTileD * s;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || j >= (x ? nkvB : nkvA)) continue;
          if (j >= 1 && !mbar_wait_warp(&bars[B_S_FREE + x], (j - 1) & 1, abort_flag, p.status, 4)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t dQ = dQ0 + kTileD * x;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 64 head dims: 32 bytes per step
              umma_bf16_ss(tmem + kColS + 128 * x, dQ + 2 * kk, dK + 2 * kk, kIdescS,
                           kk > 0 ? 1u : 0u);
            umma_commit(&bars[B_S_FULL + x]);
            if (x == 1 || j >= nkvB) umma_commit(&bars[B_K_EMPTY + s]);
          }
          __syncwarp();
        }
        if (!ok) break;
      }
      if (j >= 1) {
        const int jj = j - 1;
        const int s = jj % kStages;
        if (!mbar_wait_warp(&bars[B_V_FULL + s], (jj / kStages) & 1, abort_flag, p.status, 13)) {
          ok = false;
          break;
        }
        const uint64_t dV = dV0 + kTileD * s;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!ok || jj >= (x ? nkvB : nkvA)) continue;
          if (!mbar_wait_warp(&bars[B_P_FULL + x], jj & 1, abort_flag, p.status, 5)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t acc0 = jj > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // K = 128 keys: 8 packed P columns, 16 V rows
              umma_bf16_ts(tmem + kColO + 64 * x, tmem + kColP + 64 * x + 8 * kk,
                           dV + 128 * kk, kIdescO, kk > 0 ? 1u : acc0);
            umma_commit(&bars[B_PV_DONE + x]);
            if (jj == (x ? nkvB : nkvA) - 1) umma_commit(&bars[B_O_FINAL + x]);
            if (x == 1 || jj >= nkvB) umma_commit(&bars[B_V_EMPTY + s]);
          }
          __syncwarp();
        }
        if (!ok) break;
      }
    }
    // Drain: every MMA issued above completes before TMEM is released.
    if (elect_one()) umma_commit(&bars[B_MMA_DONE]);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(&bars[B_MMA_DONE], 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
    }
    __syncwarp();
  } else if (warp >= 12) {
    // warp 15: no role (it completes the warpgroup for setmaxnreg)
    regs_decrease<kRegsMma>();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ RoPE warps
    regs_decrease<kRegsRotate>();
    const int r = threadIdx.x - 256;  // 0..127: tile row
    RopeRow tab;
    rope_load_row(p.rope, rowA + r, tab);
    if (mbar_wait(&bars[B_Q_FULL], 0, abort_flag, p.status, 6)) {
      rope_rotate_row(sQ, r, tab);
      rope_load_row(p.rope, rowA + kBM + r, tab);
      rope_rotate_row(sQ + kTileBytes, r, tab);
      fence_proxy_async_smem();
      mbar_arrive(&bars[B_Q_ROT]);
      rope_load_row(p.rope, r, tab);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(&bars[B_K_FULL + s], (j / kStages) & 1, abort_flag, p.status, 7)) break;
        rope_rotate_row(sK + s * kTileBytes, r, tab);
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_K_ROT + s]);
        if (j + 1 < nkv) rope_load_row(p.rope, (j + 1) * kBN + r, tab);  // next tile's table
      }
    }
  } else {
    // --------------------------------------------------------- softmax warps
    regs_increase<kRegsSoftmax>();
    const int x = warp >> 2;            // tile A (0) or B (1)
    const int wq = warp & 3;            // TMEM lane quarter
    const int r = wq * 32 + lane;       // row in tile
    const int qpos = rowA + x * kBM + r;  // position in sequence
    const int nkv_x = x ? nkvB : nkvA;
    const int diag = x ? 2 * blk + 1 : 2 * blk;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128 * x;
    const uint32_t tO = tmem + lane_base + kColO + 64 * x;
    const uint32_t tP = tmem + lane_base + kColP + 64 * x;
    const float sl2 = p.scale_log2;
    float m_ref = 0.f;  // reference max (log2 units) the P values are taken against
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv_x; ++j) {
      if (!mbar_wait_warp(&bars[B_S_FULL + x], j & 1, abort_flag, p.status, 8)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // The whole S row in one TMEM round trip; S_X is then free for Q_X K_{j+1}^T.
      uint32_t sr[128];
      tmem_ld_x32(tS + 0, sr + 0);
      tmem_ld_x32(tS + 32, sr + 32);
      tmem_ld_x32(tS + 64, sr + 64);
      tmem_ld_x32(tS + 96, sr + 96);
      tmem_ld_wait(sr + 0);
      tmem_ld_wait(sr + 32);
      tmem_ld_wait(sr + 64);
      tmem_ld_wait(sr + 96);
      tc_fence_before();
      mbar_arrive(&bars[B_S_FREE + x]);
      if (j == diag) {  // diagonal tile: keys after the query get no weight
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) sr[c] = 0xff800000u;  // -inf
      }
      // Row max of the raw scores (the scale is positive), four chains.
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 128; c += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          m4[u] = fmax3(m4[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
      // Move the reference max only when the row max outgrows it by more than
      // 2^8 (exact: O and l keep a common reference).
      const bool grow = (j == 0) || (mx > m_ref + 8.0f);
      float alpha = 1.f;
      if (grow) {
        alpha = (j == 0) ? 0.f : ex2_approx(m_ref - mx);
        m_ref = mx;
      }
      // P = 2^(x - m_ref) in bf16 pairs, computed before P_X / O_X are touched.
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
      uint64_t acc[4] = {0, 0, 0, 0};  // packed partial row sums (0 = +0.f, +0.f)
      uint32_t pw[64];
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const uint64_t t = f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                  sl2x2, negm2);
        float t0, t1;
        f2_unpack(t, t0, t1);
        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
        acc[(c >> 1) & 3] = f2_add(acc[(c >> 1) & 3], f2_pack(p0, p1));
        pw[c >> 1] = pack_bf16x2(p0, p1);
      }
      float rs0, rs1;
      f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), rs0, rs1);
      const float rs = rs0 + rs1;
      // P_X and O_X are in use by the P V of the previous tile until it
      // completes (waited every tile, so PV_DONE is never two phases behind).
      if (j > 0) {
        if (!mbar_wait_warp(&bars[B_PV_DONE + x], (j - 1) & 1, abort_flag, p.status, 9)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          uint32_t o[32];
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            tmem_ld_x32(tO + half * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st_x32(tO + half * 32, o);
            tmem_st_wait();  // the store has consumed `o` before it is reloaded
          }
        }
      }
      tmem_st_x32(tP, pw);
      tmem_st_x32(tP + 32, pw + 32);
      tmem_st_wait();
      l_sum = l_sum * alpha + rs;
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL + x]);
    }
    // ---- epilogue: O / l and LSE for rows inside the sequence -------------
    // (O_FINAL completes exactly once; PV_DONE may by now be more than one
    // phase behind this thread, so its parity cannot be used here.)
    if (ok && nkv_x > 0 && mbar_wait_warp(&bars[B_O_FINAL + x], 0, abort_flag, p.status, 11)) {
      tc_fence_after();
      uint32_t o[64];
      tmem_ld_x32(tO, o);
      tmem_ld_x32(tO + 32, o + 32);
      tmem_ld_wait(o);
      tmem_ld_wait(o + 32);
      if (qpos < len) {
        const float inv_l = 1.f / l_sum;
        const long long orow = (static_cast<long long>(start + qpos) * H + h) * kHD;
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
  if (warp == 12) {
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
  dim3 grid(p.pb.nseq * p.pb.H, (n_qtiles + 1) / 2);
  ne_attn_fwd_kernel<<<grid, fwd::kThreads, fwd::SMEM_BYTES, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace ne
