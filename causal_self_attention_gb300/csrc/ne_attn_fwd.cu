// ne_attn_fwd.cu -- forward causal self-attention with fused RoPE on sm_103a.
//
// Work item: two consecutive 128-row query tiles (A: rows 256p..256p+127, B:
// rows 256p+128..256p+255) of one (sequence, head):
//   O_m = sum_{n<=m} softmax_n(scale * q'_m . k'_n) v_n,  LSE_m = log sum exp(...)
// with q' = R(m) q, k' = R(n) k (RoPE), the scores never leaving the SM
// (tiled online softmax, as in the hand-written FlashAttention of the
// NanoEuler Show HN page, paragraph 2; causality as in "Tiny Hackable CUDA",
// section 3).  Both tiles share every K'/V tile, and while one tile's
// softmax runs the tensor core works on the other tile's MMAs.
//
// RoPE: each query tile is used by one item only and is rotated in shared
// memory right after its TMA load.  A key tile is used by every query tile at
// or after it; the keys are rotated either in shared memory by every item
// that uses them (kRotateK = 1, short sequences: no extra pass), or once
// per call by a small pass that runs first (ne_attn_rope_rows_kernel,
// k' = R(n) k, bf16; kRotateK = 0, long sequences, where rotating each key
// tile several times -- its table loads -- paces the kernel).  The training
// forward rotates queries and keys in that pass, into buffers the caller
// keeps for the backward, and the kernel then rotates nothing (kRotateQ = 0).
//
// The kernel is persistent: one CTA per SM walks the items (longest first,
// dealt out in a snake order over the CTAs), keeping its TMEM, barriers and
// K/V rings across items, so that the next item's Q load and RoPE overlap the
// current item's last tiles and its epilogue.  Q is double-buffered.
//
// Warp roles (512 threads, registers re-split per warpgroup with setmaxnreg):
//   warps 0-3   softmax A: thread t owns row t of tile A (TMEM lane t), 176 regs
//   warps 4-7   softmax B: same for tile B
//   warps 8-11  rotate: RoPE on each item's Q_A, Q_B in smem (and, with
//               rotate_k, on every K tile it uses), 104 regs
//   warp 12     MMA: allocates TMEM; one elected lane issues S_X = Q_X K^T
//   warp 13     TMA: lane 0 loads each item's Q_A, Q_B and the K' ring (5 stages)
//   warp 14     TMA: lane 0 loads the V ring (5 stages)
//   warp 15     MMA: one elected lane issues O_X += P_X V; warps 12-15 run at
//               56 regs
// TMEM columns: S_A 0-127, S_B 128-255, O_A 256-319, O_B 320-383,
// P_A 384-447, P_B 448-511 (bf16 pairs: P is the TMEM A operand of P V).
// A softmax thread loads its whole S row with one TMEM round trip and frees
// S_X at once, so the next S_X = Q_X K^T overlaps the exponentials; the
// reference max moves only when the row max grows by more than 2^8 (exact: O
// and l keep a common reference).
// Key tiles entirely above the diagonal are never loaded or computed.
//
// Barrier phases: the K and V rings count K tiles over all items of the CTA;
// S_FULL / S_FREE / P_FULL / PV_DONE of tile X count the steps of tile X over
// all items; Q_* (per Q buffer), O_FINAL and O_FREE count items.
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace fwd {

constexpr int kThreads = 512;
// Registers per thread of each warpgroup after setmaxnreg (launch: 128).
constexpr uint32_t kRegsSoftmax = 176, kRegsRotate = 104, kRegsMma = 56;
static_assert(valid_reg_split(kRegsSoftmax, kRegsRotate, kRegsMma), "register split");
constexpr int kStages = 5;                            // K ring and V ring
constexpr int OFF_Q = 0;                              // 2 buffers x (Q_A, Q_B)
constexpr int OFF_K = OFF_Q + 4 * kTileBytes;         // kStages
constexpr int OFF_V = OFF_K + kStages * kTileBytes;   // kStages
constexpr int OFF_BAR = OFF_V + kStages * kTileBytes;
constexpr int kBarBytes = 512;  // mbarriers, TMEM address, abort flag
constexpr int SMEM_BYTES = OFF_BAR + kBarBytes + 1024;  // + slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "more shared memory than an sm_103 CTA may have");

enum Bar {
  B_Q_FULL = 0,                       // per Q buffer
  B_Q_ROT = B_Q_FULL + 2,
  B_Q_EMPTY = B_Q_ROT + 2,
  B_K_FULL = B_Q_EMPTY + 2,           // kStages
  B_K_ROT = B_K_FULL + kStages,       // kStages (rotate_k only)
  B_K_EMPTY = B_K_ROT + kStages,      // kStages
  B_V_FULL = B_K_EMPTY + kStages,     // kStages
  B_V_EMPTY = B_V_FULL + kStages,     // kStages
  B_S_FULL = B_V_EMPTY + kStages,     // per tile X
  B_S_FREE = B_S_FULL + 2,
  B_P_FULL = B_S_FREE + 2,
  B_PV_DONE = B_P_FULL + 2,
  B_O_FINAL = B_PV_DONE + 2,          // per tile: the item's last P V completed
  B_O_FREE = B_O_FINAL + 2,           // per tile: the epilogue has read O_X
  B_OST_FULL = B_O_FREE + 2,          // per tile: O_X (bf16) staged in its Q slot
  B_MMA_DONE = B_OST_FULL + 2,        // per issuing warp (S, P V)
  B_COUNT = B_MMA_DONE + 2
};
static_assert(8 * B_COUNT + 8 <= kBarBytes, "barrier region overflow");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S_X at 128 * X
constexpr uint32_t kColO = 256;  // O_X at 256 + 64 * X
constexpr uint32_t kColP = 384;  // P_X at 384 + 64 * X

constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);  // Q K^T
constexpr uint32_t kIdescO = make_idesc_bf16(128, 64, false, true);    // P V (V MN-major)

// One work item: block `blk` of 256 query rows of (sequence seq, head h).
struct Item {
  int seq, h, blk;
  int start, len;  // the sequence's first row in the packed tensors, its length
  int rowA;        // first row of tile A in the sequence
  bool hasB;       // tile B has rows inside the sequence
  int nkvA, nkvB, nkv;  // key tiles of A, of B, and of the item (causal)
};

// Item `r` of the longest-first order: all blocks with the highest index
// first (they have the most key tiles), then the next lower, ...  Returns
// false for an empty item (the sequence has no such block, or a bad
// cu_seqlens entry, which is reported once).
__device__ __forceinline__ bool get_item(const FwdParams& p, int nblk, int r, Item& it,
                                         bool report) {
  const int n_sh = p.pb.nseq * p.pb.H;
  const int sh = r % n_sh;
  it.blk = nblk - 1 - r / n_sh;
  it.seq = sh / p.pb.H;
  it.h = sh % p.pb.H;
  if (!seq_bounds(p.pb, it.seq, it.start, it.len, (report && it.blk == 0) ? p.status : nullptr))
    return false;
  it.rowA = 2 * it.blk * kBM;
  if (it.rowA >= it.len) return false;
  it.hasB = it.rowA + kBM < it.len;
  it.nkvA = 2 * it.blk + 1;  // key tiles 0..2blk for A, 0..2blk+1 for B
  it.nkvB = it.hasB ? 2 * it.blk + 2 : 0;
  it.nkv = it.hasB ? it.nkvB : it.nkvA;
  return true;
}

}  // namespace fwd

// Grid: G persistent CTAs; nblk = 256-row blocks of the longest sequence.
// kRotateK: the K tiles are rotated in smem by the rotate warps (short
// sequences); otherwise they come pre-rotated and the O tiles are written by
// TMA from the Q buffer (long sequences).  kRotateQ: the Q tiles are rotated
// in smem (always, except for callers that pass q' = R(m) q already rotated,
// e.g. by the QKV projection's epilogue).  Separate instantiations, so that
// each compiles only its own epilogue (registers are tight in the softmax
// warps).
template <bool kRotateK, bool kRotateQ>
__global__ void __launch_bounds__(fwd::kThreads, 1)
    ne_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmO, const FwdParams p, int nblk) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);

  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int n_items = nblk * p.pb.nseq * p.pb.H;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_Q_FULL + b], 1);
      mbar_init(&bars[B_Q_ROT + b], 128);
      // The item's last S MMA and, when O tiles are staged in the Q buffer
      // (pre-rotated keys), its O tile stores.
      mbar_init(&bars[B_Q_EMPTY + b], kRotateK ? 1 : 2);
    }
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
      mbar_init(&bars[B_O_FREE + x], 128);
      mbar_init(&bars[B_OST_FULL + x], 128);
    }
    mbar_init(&bars[B_MMA_DONE], 1);
    mbar_init(&bars[B_MMA_DONE + 1], 1);
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
  pdl_wait();  // whatever the stream ran before (e.g. the kernel that wrote q, k, v) has completed
  pdl_launch_dependents();

  uint8_t* sQ = smem + OFF_Q;  // buffer b: Q_A at 2b tiles, Q_B at 2b + 1
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  // The items of this CTA, in order (the same sequence in every role).
#define NE_FOR_EACH_ITEM(it)                                                        \
  for (int k_ = 0, r_ = dealt_item(nullptr, p.compact, 0, cta, G, n_items); r_ < n_items;       \
       ++k_, r_ = dealt_item(nullptr, p.compact, k_, cta, G, n_items))                             \
    if (Item it; get_item(p, nblk, r_, it, threadIdx.x == 0))

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
      if (isK) tma_prefetch_desc(&tmQ);
      bool ok = true;
      int g = 0;   // K (or V) tiles loaded so far by this CTA
      int nq = 0;  // items whose Q has been loaded
      NE_FOR_EACH_ITEM(it) {
        if (!ok) break;
        if (isK) {
          const int b = nq & 1;
          if (nq >= 2 && !mbar_wait(&bars[B_Q_EMPTY + b], ((nq - 2) >> 1) & 1, abort_flag,
                                    p.status, 14)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[B_Q_FULL + b], 2 * kTileBytes);
          tma_load_3d(sQ + 2 * b * kTileBytes, &tmQ, &bars[B_Q_FULL + b], 0, it.h,
                      it.start + it.rowA);
          tma_load_3d(sQ + (2 * b + 1) * kTileBytes, &tmQ, &bars[B_Q_FULL + b], 0, it.h,
                      it.start + it.rowA + kBM);
          ++nq;
        }
        for (int j = 0; j < it.nkv; ++j, ++g) {
          const int s = g % kStages;
          if (g >= kStages &&
              !mbar_wait(&empty[s], ((g - kStages) / kStages) & 1, abort_flag, p.status,
                         isK ? 1 : 12)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kTileBytes);
          tma_load_3d(ring + s * kTileBytes, tm, &full[s], 0, it.h, it.start + j * kBN);
        }
      }
      if (!ok || *abort_flag) {
        // Let the copies still in flight land before the CTA exits: every
        // issued load completes its FULL barrier phase.
        for (int s = 0; s < kStages; ++s) {
          if (g > s) {
            const int last = s + ((g - 1 - s) / kStages) * kStages;  // last tile loaded into s
            const long long t0 = clock64();
            while (!mbar_try_wait(&full[s], (last / kStages) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
        }
        if (isK)
          for (int q = (nq >= 2 ? nq - 2 : 0); q < nq; ++q) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[B_Q_FULL + (q & 1)], (q >> 1) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
      }
    } else if (!kRotateK && warp == 14 && lane == 1) {
      // O tile stores (pre-rotated keys only): once a tile's softmax threads
      // have staged its bf16 O in the tile's own Q slot (no S MMA reads it any
      // more), store it with TMA; when both tiles of the item are stored
      // (their smem read), hand the Q buffer back to the loader.  Partial
      // tiles (rows past the sequence) and fp32 output are written by the
      // softmax threads.  With in-kernel key rotation the Q buffer goes back
      // at the item's last S MMA (the rotate warps need the next items' Q
      // early) and every row is written by its softmax thread.
      tma_prefetch_desc(&tmO);
      int nq = 0, nst[2] = {0, 0};
      NE_FOR_EACH_ITEM(it) {
        const int b = nq & 1;
        bool ok = true;
        for (int x = 0; x < 2 && ok; ++x) {
          if (x == 1 && !it.hasB) continue;
          if (!(ok = mbar_wait(&bars[B_OST_FULL + x], nst[x] & 1, abort_flag, p.status, 16))) break;
          ++nst[x];
          const int row0 = it.rowA + x * kBM;
          if (!p.out_f32 && row0 + kBM <= it.len)
            tma_store_3d(&tmO, sQ + (2 * b + x) * kTileBytes, 0, it.h, it.start + row0);
        }
        if (!ok) break;
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(&bars[B_Q_EMPTY + b]);
        ++nq;
      }
      bulk_wait_group0();  // the stores have completed before the kernel ends
    }
  } else if (warp == 12 || warp == 15) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 12 issues S_X = Q_X K^T and warp 15 issues O_X += P_X V, both
    // walking the same items; each commit sits on the warp whose MMAs it
    // tracks (a commit covers only the MMAs its own thread issued).  The whole
    // warp runs the loop and waits; the elected lane issues each group of MMAs
    // together with its commits.  Shared-memory descriptors are built once: a
    // K step, a tile or a ring stage only adds a constant to the start-address
    // field (16-byte units).
    regs_decrease<kRegsMma>();
    const bool isS = (warp == 12);
    constexpr uint64_t kTileD = kTileBytes >> 4;
    const uint64_t dQ0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);          // Q K-major
    const uint64_t dK0 = make_sdesc_sw128(smem_u32(sK), 16, 1024);          // K K-major
    const uint64_t dV0 = make_sdesc_sw128(smem_u32(sV), kTileBytes, 1024);  // V MN-major
    bool ok = true;
    int g = 0;                 // K / V tiles consumed
    int nq = 0;                // items started (Q buffer and phase)
    int cnt[2] = {0, 0};       // steps of tile X over all items
    int nit[2] = {0, 0};       // items in which tile X took part
    NE_FOR_EACH_ITEM(it) {
      if (!ok) break;
      const int b = nq & 1;
      const int g0 = g;
      if (isS) {
        ok = mbar_wait_warp(&bars[B_Q_ROT + b], (nq >> 1) & 1, abort_flag, p.status, 2);
        for (int j = 0; ok && j < it.nkv; ++j) {
          const int gj = g0 + j, s = gj % kStages;
          if (!mbar_wait_warp(&bars[(kRotateK ? B_K_ROT : B_K_FULL) + s], (gj / kStages) & 1,
                              abort_flag, p.status, 3)) {
            ok = false;
            break;
          }
          const uint64_t dK = dK0 + kTileD * s;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok || j >= (x ? it.nkvB : it.nkvA)) continue;
            const int c = cnt[x] + j;
            if (c >= 1 && !mbar_wait_warp(&bars[B_S_FREE + x], (c - 1) & 1, abort_flag, p.status, 4)) {
              ok = false;
              continue;
            }
            tc_fence_after();
            if (elect_one()) {
              // Descriptors formed at issue, not hoisted out of the loop.
              const uint64_t dQ = opaque_u64(dQ0) + kTileD * (2 * b + x);
              const uint64_t dKs = opaque_u64(dK);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K = 64 head dims: 32 bytes per step
                umma_bf16_ss(tmem + kColS + 128 * x, dQ + 2 * kk, dKs + 2 * kk, kIdescS,
                             kk > 0 ? 1u : 0u);
              umma_commit(&bars[B_S_FULL + x]);
              if (x == 1 || j >= it.nkvB) umma_commit(&bars[B_K_EMPTY + s]);
              if (j == it.nkv - 1 && (x == 1 || !it.hasB)) umma_commit(&bars[B_Q_EMPTY + b]);
            }
            __syncwarp();
          }
        }
      } else {
        for (int jj = 0; ok && jj < it.nkv; ++jj) {
          const int gj = g0 + jj, s = gj % kStages;
          if (!mbar_wait_warp(&bars[B_V_FULL + s], (gj / kStages) & 1, abort_flag, p.status, 13)) {
            ok = false;
            break;
          }
          const uint64_t dV = dV0 + kTileD * s;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok || jj >= (x ? it.nkvB : it.nkvA)) continue;
            const int c = cnt[x] + jj;
            if (!mbar_wait_warp(&bars[B_P_FULL + x], c & 1, abort_flag, p.status, 5)) {
              ok = false;
              continue;
            }
            // The first P V of an item overwrites O_X: the previous item's
            // epilogue must have read it.
            if (jj == 0 && nit[x] >= 1 &&
                !mbar_wait_warp(&bars[B_O_FREE + x], (nit[x] - 1) & 1, abort_flag, p.status, 15)) {
              ok = false;
              continue;
            }
            tc_fence_after();
            if (elect_one()) {
              const uint32_t acc0 = jj > 0 ? 1u : 0u;
              const uint64_t dVs = opaque_u64(dV);  // formed at issue, not hoisted
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)  // K = 128 keys: 8 packed P columns, 16 V rows
                umma_bf16_ts(tmem + kColO + 64 * x, tmem + kColP + 64 * x + 8 * kk,
                             dVs + 128 * kk, kIdescO, kk > 0 ? 1u : acc0);
              umma_commit(&bars[B_PV_DONE + x]);
              if (jj == (x ? it.nkvB : it.nkvA) - 1) umma_commit(&bars[B_O_FINAL + x]);
              if (x == 1 || jj >= it.nkvB) umma_commit(&bars[B_V_EMPTY + s]);
            }
            __syncwarp();
          }
        }
      }
      g = g0 + it.nkv;
      cnt[0] += it.nkvA;
      cnt[1] += it.nkvB;
      nit[0] += 1;
      nit[1] += it.hasB ? 1 : 0;
      ++nq;
    }
    // Drain: every MMA this warp issued completes before TMEM is released.
    uint64_t* done = &bars[B_MMA_DONE + (isS ? 0 : 1)];
    if (elect_one()) umma_commit(done);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(done, 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ RoPE warps
    regs_decrease<kRegsRotate>();
    const int r = threadIdx.x - 256;  // 0..127: tile row
    RopeRow tab;
    bool ok = true;
    int g = 0, nq = 0;
    NE_FOR_EACH_ITEM(it) {
      if (!ok) break;
      const int b = nq & 1;
      if constexpr (kRotateQ) rope_load_row(p.rope, it.rowA + r, tab);
      if (!(ok = mbar_wait(&bars[B_Q_FULL + b], (nq >> 1) & 1, abort_flag, p.status, 6))) break;
      if constexpr (kRotateQ) {
        rope_rotate_row(sQ + 2 * b * kTileBytes, r, tab);
        rope_load_row(p.rope, it.rowA + kBM + r, tab);
        rope_rotate_row(sQ + (2 * b + 1) * kTileBytes, r, tab);
        fence_proxy_async_smem();
      }
      mbar_arrive(&bars[B_Q_ROT + b]);
      ++nq;
      if (!kRotateK) continue;  // the keys come pre-rotated
      rope_load_row(p.rope, r, tab);
      for (int j = 0; j < it.nkv; ++j, ++g) {
        const int s = g % kStages;
        if (!(ok = mbar_wait(&bars[B_K_FULL + s], (g / kStages) & 1, abort_flag, p.status, 7)))
          break;
        rope_rotate_row(sK + s * kTileBytes, r, tab);
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_K_ROT + s]);
        if (j + 1 < it.nkv) rope_load_row(p.rope, (j + 1) * kBN + r, tab);  // next tile's table
      }
    }
  } else {
    // --------------------------------------------------------- softmax warps
    regs_increase<kRegsSoftmax>();
    const int x = warp >> 2;            // tile A (0) or B (1)
    const int wq = warp & 3;            // TMEM lane quarter
    const int r = wq * 32 + lane;       // row in tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128 * x;
    const uint32_t tO = tmem + lane_base + kColO + 64 * x;
    const uint32_t tP = tmem + lane_base + kColP + 64 * x;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int cnt = 0;  // steps of this tile over all items
    int nit = 0;  // items in which this tile took part
    int nq = 0;   // items (the Q buffer of item nq is nq & 1)
    NE_FOR_EACH_ITEM(it) {
      if (!ok) break;
      const int nkv_x = x ? it.nkvB : it.nkvA;
      if constexpr (!kRotateK) ++nq;
      if (nkv_x == 0) continue;  // tile B outside the sequence
      const int diag = x ? 2 * it.blk + 1 : 2 * it.blk;
      float m_ref = 0.f;  // reference max (log2 units) the P values are taken against
      float l_sum = 0.f;
      for (int j = 0; j < nkv_x; ++j) {
        const int c = cnt + j;
        if (!(ok = mbar_wait_warp(&bars[B_S_FULL + x], c & 1, abort_flag, p.status, 8))) break;
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
          for (int cc = 0; cc < 128; ++cc)
            if (cc > r) sr[cc] = 0xff800000u;  // -inf
        }
        // Row max of the raw scores (the scale is positive), four chains.
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cc = 0; cc < 128; cc += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            m4[u] = fmax3(m4[u], __uint_as_float(sr[cc + 2 * u]),
                          __uint_as_float(sr[cc + 2 * u + 1]));
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
        // Move the reference max only when the row max outgrows it by more
        // than 2^8 (exact: O and l keep a common reference).
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
        for (int cc = 0; cc < 128; cc += 2) {
          const uint64_t t = f2_fma(f2_pack(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])),
                                    sl2x2, negm2);
          float t0, t1;
          f2_unpack(t, t0, t1);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
          acc[(cc >> 1) & 3] = f2_add(acc[(cc >> 1) & 3], f2_pack(p0, p1));
          pw[cc >> 1] = pack_bf16x2(p0, p1);
        }
        float rs0, rs1;
        f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), rs0, rs1);
        const float rs = rs0 + rs1;
        // P_X and O_X are in use by the P V of the previous tile until it
        // completes (waited every tile, so PV_DONE is never two phases behind;
        // at an item's first tile the previous item's epilogue has already
        // seen its last P V complete).
        if (j > 0) {
          if (!(ok = mbar_wait_warp(&bars[B_PV_DONE + x], (c - 1) & 1, abort_flag, p.status, 9)))
            break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, grow)) {
            uint32_t o[32];
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              tmem_ld_x32(tO + half * 32, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) o[cc] = __float_as_uint(__uint_as_float(o[cc]) * alpha);
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
      if (!ok) break;
      cnt += nkv_x;
      // ---- epilogue: O / l and LSE for rows inside the sequence -----------
      if (!(ok = mbar_wait_warp(&bars[B_O_FINAL + x], nit & 1, abort_flag, p.status, 11))) break;
      ++nit;
      // The item's placement is derived again here from an opaque copy of its
      // index, so that none of it stays live (in registers or spilled) through
      // the loop above.
      Item e;
      get_item(p, nblk, opaque_int(r_), e, false);
      const int erow = e.rowA + x * kBM + r;
      tc_fence_after();
      uint32_t o[64];
      tmem_ld_x32(tO, o);
      tmem_ld_x32(tO + 32, o + 32);
      tmem_ld_wait(o);
      tmem_ld_wait(o + 32);
      tc_fence_before();
      mbar_arrive(&bars[B_O_FREE + x]);  // the next item's first P V may overwrite O_X
      if constexpr (kRotateK) {
        // Every row written by its own thread.
        if (erow < e.len) {
          const float inv_l = 1.f / l_sum;
          const long long orow = (static_cast<long long>(e.start + erow) * p.pb.H + e.h) * kHD;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              dst[cc] = make_float4(__uint_as_float(o[4 * cc + 0]) * inv_l,
                                    __uint_as_float(o[4 * cc + 1]) * inv_l,
                                    __uint_as_float(o[4 * cc + 2]) * inv_l,
                                    __uint_as_float(o[4 * cc + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow);
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[8 * cc + 0]) * inv_l, __uint_as_float(o[8 * cc + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(o[8 * cc + 2]) * inv_l, __uint_as_float(o[8 * cc + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(o[8 * cc + 4]) * inv_l, __uint_as_float(o[8 * cc + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(o[8 * cc + 6]) * inv_l, __uint_as_float(o[8 * cc + 7]) * inv_l);
              dst[cc] = w;
            }
          }
          // LSE in natural-log units: (m_ref + log2 l) * ln 2.
          p.lse[lse_index(p.pb, e.h, e.seq, e.start, erow)] =
              (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
        }
      } else {
        const float inv_l = 1.f / l_sum;
        const long long orow = (static_cast<long long>(e.start + erow) * p.pb.H + e.h) * kHD;
        if (p.out_f32) {
          if (erow < e.len) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow);
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              dst[cc] = make_float4(__uint_as_float(o[4 * cc + 0]) * inv_l,
                                    __uint_as_float(o[4 * cc + 1]) * inv_l,
                                    __uint_as_float(o[4 * cc + 2]) * inv_l,
                                    __uint_as_float(o[4 * cc + 3]) * inv_l);
          }
        } else {
          // A whole tile goes, row r in bf16, into the swizzled Q slot of this
          // tile (item nq - 1's buffer), and warp 14, lane 1 stores it with
          // TMA; the sequence's last, partial tile is written one row per
          // thread.
          const bool whole = e.rowA + x * kBM + kBM <= e.len;
          uint8_t* slot = sQ + (2 * (opaque_int(nq - 1) & 1) + x) * kTileBytes;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow);
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * cc + 0]) * inv_l, __uint_as_float(o[8 * cc + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * cc + 2]) * inv_l, __uint_as_float(o[8 * cc + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * cc + 4]) * inv_l, __uint_as_float(o[8 * cc + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * cc + 6]) * inv_l, __uint_as_float(o[8 * cc + 7]) * inv_l);
            if (whole)
              *reinterpret_cast<uint4*>(slot + sw128_offset(r, cc)) = w;
            else if (erow < e.len)
              dst[cc] = w;
          }
          if (whole) fence_proxy_async_smem();
        }
        mbar_arrive(&bars[B_OST_FULL + x]);
        // LSE in natural-log units: (m_ref + log2 l) * ln 2.
        if (erow < e.len)
          p.lse[lse_index(p.pb, e.h, e.seq, e.start, erow)] =
              (m_ref + __log2f(l_sum)) * 0.69314718055994531f;
      }
    }
  }
#undef NE_FOR_EACH_ITEM

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Rotation pass: xr = R(n) x for every row n of every sequence (positions
// restart at 0 per sequence), for the keys alone (k' of a long-sequence
// forward) or for queries and keys together (q', k' of the training forward),
// bf16 in and out, with the fp32 rule of the in-tile rotation (lo = fma(x_i,
// c, -(x_{i+32} s)), hi = fma(x_{i+32}, c, x_i s), round to nearest even) and
// the same table, so the attention kernel multiplies bitwise the operands an
// in-tile rotation would have produced.
// Grid (blocks of 256 items, sequences, tensors); an item is (row, head, part): part c
// rotates the 16-byte chunk c (dims 8c..8c+7) against chunk c + 4 (dims
// 32+8c..32+8c+7), so a warp moves eight whole 128-byte rows.
// ---------------------------------------------------------------------------
constexpr int kRopeThreads = 256, kRopeParts = 4;

__global__ void __launch_bounds__(kRopeThreads)
    ne_attn_rope_rows_kernel(const __nv_bfloat16* __restrict__ x0, __nv_bfloat16* __restrict__ xr0,
                             const __nv_bfloat16* __restrict__ x1, __nv_bfloat16* __restrict__ xr1,
                             const Problem pb, RopeTable rope) {
  pdl_wait();  // the kernel that wrote q, k (and anything before it) has completed
  const __nv_bfloat16* __restrict__ x = blockIdx.z ? x1 : x0;
  __nv_bfloat16* __restrict__ xr = blockIdx.z ? xr1 : xr0;
  const int seq = blockIdx.y;
  int start, len;
  if (!seq_bounds(pb, seq, start, len, nullptr)) return;
  const int H = pb.H;
  const long long w = static_cast<long long>(blockIdx.x) * kRopeThreads + threadIdx.x;
  if (w < static_cast<long long>(len) * H * kRopeParts) {
    const int c = static_cast<int>(w % kRopeParts);
    const int rh = static_cast<int>(w / kRopeParts);  // (row, head) pairs fit in 32 bits
    const int pos = rh / H, h = rh - pos * H;
    const long long row = (static_cast<long long>(start + pos) * H + h) * kHD;
    const uint4 lo = __ldg(reinterpret_cast<const uint4*>(x + row) + c);
    const uint4 hi = __ldg(reinterpret_cast<const uint4*>(x + row) + c + 4);
    const float4* cs =
        reinterpret_cast<const float4*>(rope.cs + static_cast<long long>(pos) * 32 + 8 * c);
    uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
    uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 t = __ldg(cs + u);  // (cos, sin) of dims 8c + 2u and 8c + 2u + 1
      const float a0 = bf16lo_to_f32(wl[u]), a1 = bf16hi_to_f32(wl[u]);
      const float b0 = bf16lo_to_f32(wh[u]), b1 = bf16hi_to_f32(wh[u]);
      const float lo0 = __fmaf_rn(a0, t.x, -__fmul_rn(b0, t.y));
      const float hi0 = __fmaf_rn(b0, t.x, __fmul_rn(a0, t.y));
      const float lo1 = __fmaf_rn(a1, t.z, -__fmul_rn(b1, t.w));
      const float hi1 = __fmaf_rn(b1, t.z, __fmul_rn(a1, t.w));
      wl[u] = pack_bf16x2(lo0, lo1);
      wh[u] = pack_bf16x2(hi0, hi1);
    }
    reinterpret_cast<uint4*>(xr + row)[c] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    reinterpret_cast<uint4*>(xr + row)[c + 4] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  }
  pdl_launch_dependents();
}

// x1, xr1: a second tensor rotated by the same launch, or null.
cudaError_t launch_rope_rows(const __nv_bfloat16* x0, __nv_bfloat16* xr0,
                             const __nv_bfloat16* x1, __nv_bfloat16* xr1, const Problem& pb,
                             const RopeTable& rope, cudaStream_t stream) {
  const long long items = static_cast<long long>(pb.max_len) * pb.H * kRopeParts;
  dim3 grid(static_cast<unsigned>((items + kRopeThreads - 1) / kRopeThreads), pb.nseq,
            x1 ? 2 : 1);
  return launch_pdl(ne_attn_rope_rows_kernel, grid, dim3(kRopeThreads), 0, stream, x0, xr0, x1,
                    xr1, pb, rope);
}

cudaError_t launch_fwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmO, const FwdParams& p, int n_qtiles,
                       cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_attn_fwd_kernel<true, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fwd::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ne_attn_fwd_kernel<false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ne_attn_fwd_kernel<false, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // One persistent CTA per SM (at most one per item).
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sm_count[dev]) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int nblk = (n_qtiles + 1) / 2;
  const long long n_items = static_cast<long long>(nblk) * p.pb.nseq * p.pb.H;
  const int G = static_cast<int>(n_items < sm_count[dev] ? n_items : sm_count[dev]);
  if (p.rotate_k)
    return launch_pdl(ne_attn_fwd_kernel<true, true>, dim3(G), dim3(fwd::kThreads),
                      fwd::SMEM_BYTES, stream, tmQ, tmK, tmV, tmO, p, nblk);
  if (p.rotate_q)
    return launch_pdl(ne_attn_fwd_kernel<false, true>, dim3(G), dim3(fwd::kThreads),
                      fwd::SMEM_BYTES, stream, tmQ, tmK, tmV, tmO, p, nblk);
  return launch_pdl(ne_attn_fwd_kernel<false, false>, dim3(G), dim3(fwd::kThreads),
                    fwd::SMEM_BYTES, stream, tmQ, tmK, tmV, tmO, p, nblk);
}

}  // namespace ne
