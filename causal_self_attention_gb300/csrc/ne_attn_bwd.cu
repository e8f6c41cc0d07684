// ne_attn_bwd.cu -- backward of causal self-attention with RoPE, sm_103a.
//
// Three kernels on one stream, each launched with programmatic dependent
// launch so that its CTAs set up while the previous kernel drains (gradients
// hand-derived, no autograd, as the NanoEuler Show HN page, paragraph 2,
// describes for its engine):
//   1. preprocess, once per element: D_m = dO_m . O_m (fp32, [H, N_tot]); zero
//      the fp32 dQ' accumulator; and q' = R(m) q, k' = R(n) k into bf16
//      workspace buffers with the forward's fp32 rule, so the main kernel
//      multiplies exactly the operands the forward did and rotates nothing
//      (a query tile is used by every key tile at or before it: rotating it
//      there would repeat the work once per key tile).  When the caller
//      passes q', k' (the training pair) nothing is rotated, and a
//      persistent form streams O and dO through shared memory instead;
//   2. main: persistent, one CTA per SM; each walks its units (128-key tile
//      j of one (sequence, head)) and, per unit, the query tiles i >= j,
//      recomputing P from the saved LSE:
//        S^T  = K' Q'^T,  P^T = exp(scale S^T - LSE),  dP^T = V dO^T,
//        dS^T = P^T o (dP^T - D),
//        dV  += P^T dO (P^T from TMEM),  dK' += dS^T Q',  dQ'_i = dS K'
//        (-> bulk tensor reduce-add),
//      and at the end of each unit writes dV and scale * dK' (bf16).  K' is
//      double-buffered across units, so the next unit's K' is loaded while
//      the current unit runs; V is reloaded as soon as the unit's last dP^T
//      has read it;
//   3. postprocess: dQ = scale * R(m)^T dQ' (bf16), and dK = R(n)^T (scale dK')
//      in place (rotating dK here rather than at the end of each unit keeps
//      table loads off the unit boundary, where they held up the next unit).
//
// Main-kernel warp roles (512 threads, registers re-split per warpgroup):
//   warps 0-3   row terms and dQ': stage -LSE_i and -D_i two tiles ahead;
//               after tile i, move dQ'_i (64 fp32 columns per query row) from TMEM to two swizzled staging buffers and
//               issue their bulk reduce-adds
//   warps 4-7   softmax, query columns 0-63 of the tile (thread t: key row t)
//   warps 8-11  softmax, query columns 64-127; a softmax thread reads its S^T
//               and dP^T half-rows in one TMEM round trip and frees them at
//               once, so the next tile's S^T/dP^T MMAs overlap its math; it
//               writes P^T to TMEM (A operand of dV) and dS^T to smem
//   warp 12     MMA: allocates TMEM; its elected lane issues dV, dK' and dQ'
//               of every tile (24 MMAs)
//   warp 13     TMA: lane 0 loads Q'_i, dO_i (3 stages, continuing across units)
//   warp 14     MMA: its elected lane issues S^T and dP^T of every tile (8
//               MMAs).  Two issuing warps: one warp issuing all 32 MMAs of a
//               tile was measured to pace the whole loop (its instructions
//               compete with the softmax warps for issue slots).
//   warp 15     TMA: lane 0 loads each unit's K'_j into the K' buffer the
//               unit before the previous one has released, and V_j once the
//               previous unit's last dP^T has completed
// TMEM columns: S^T 0-127, dP^T 128-255, dV 256-319, dK' 320-383, dQ' 384-447,
// P^T 448-511 (bf16 pairs).
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

namespace bwd {

constexpr int kThreads = 512;
// Registers per thread of each warpgroup after setmaxnreg (launch: 128).
constexpr uint32_t kRegsSoftmax = 168, kRegsDrain = 104, kRegsMma = 72;
static_assert(valid_reg_split(kRegsSoftmax, kRegsDrain, kRegsMma), "register split");
constexpr int kQStages = 3;                          // Q_i / dO_i ring depth
constexpr int OFF_K = 0;                               // 2 buffers (units alternate)
constexpr int OFF_V = OFF_K + 2 * kTileBytes;
constexpr int OFF_Q = OFF_V + kTileBytes;              // kQStages
constexpr int OFF_DO = OFF_Q + kQStages * kTileBytes;  // kQStages
constexpr int OFF_DST = OFF_DO + kQStages * kTileBytes;  // dS^T: 2 blocks of 64 queries
constexpr int OFF_DQ = OFF_DST + 2 * kTileBytes;         // dQ' staging: 2 x [128][32] fp32, SW128
// Row terms of the query tiles, staged kRowSlots - 1 tiles ahead of use.
constexpr int kRowSlots = 4;
constexpr int OFF_LSE = OFF_DQ + 2 * kTileBytes;          // kRowSlots x 128 fp32: -LSE (log2 units)
constexpr int OFF_DEL = OFF_LSE + kRowSlots * 128 * 4;  // kRowSlots x 128 fp32: -D
constexpr int OFF_BAR = OFF_DEL + kRowSlots * 128 * 4;
constexpr int kBarBytes = 512;  // mbarriers, TMEM address, abort flag
constexpr int SMEM_BYTES = OFF_BAR + kBarBytes + 1024;  // + slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "more shared memory than an sm_103 CTA may have");

enum Bar {
  B_K_FULL = 0,                          // 2 (per K' buffer): K' landed
  B_K_EMPTY = B_K_FULL + 2,              // 2: both issuing warps done with the buffer's K'
  B_V_FULL = B_K_EMPTY + 2,              // per unit: V landed
  B_V_EMPTY,                             // per unit: the unit's last dP^T completed
  B_EPI_FULL,                            // per unit: dV, scale dK' staged in the dS^T buffer
  B_EPI_READ,                            // per unit: their tile stores have read the buffer
  B_QDO_FULL,                            // kQStages
  B_ROW_FULL = B_QDO_FULL + kQStages,    // kRowSlots: -LSE_i, -D_i staged
  B_ROW_EMPTY = B_ROW_FULL + kRowSlots,  // kRowSlots: every softmax warp has read them
  B_QDO_EMPTY = B_ROW_EMPTY + kRowSlots, // kQStages
  B_S_FULL = B_QDO_EMPTY + kQStages,
  B_S_FREE,
  B_DS_FULL,
  B_PDS_FREE,
  B_DQ_FULL,
  B_DQ_FREE,
  B_MMA_DONE,                            // warp 12's MMAs all completed
  B_SDP_DONE,                            // warp 14's MMAs all completed
  B_COUNT
};
static_assert(8 * B_COUNT + 8 <= kBarBytes, "barrier region overflow");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384,
                   kColPT = 448;

constexpr uint32_t kIdescNN = make_idesc_bf16(128, 128, false, false);  // S^T, dP^T
constexpr uint32_t kIdescKM = make_idesc_bf16(128, 64, false, true);    // dV, dK
constexpr uint32_t kIdescMM = make_idesc_bf16(128, 64, true, true);     // dQ

constexpr int kPreRows = 16;   // rows per CTA of the preprocess

}  // namespace bwd

// ---------------------------------------------------------------------------
// 1. preprocess of the plain pair (q, k un-rotated).  Grid (row blocks of
//    kPreRows, sequences); 8 threads per (row, head) pair.  Thread `part`
//    (0..7) of a pair:
//      - multiplies its 8 of the 64 products dO . O (summed over the 8
//        threads by shuffles) -> D_m;
//      - zeroes its 8 floats of the dQ' accumulator row;
//      - parts 0-3 rotate chunk `part` of q (dims 8c..8c+7) against chunk
//        `part` + 4 into q', parts 4-7 the same chunks of k into k', with the
//        fp32 rule of the forward's in-tile rotation (bitwise the same values).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    ne_attn_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ q,
                                  const __nv_bfloat16* __restrict__ k,
                                  const __nv_bfloat16* __restrict__ out,
                                  const __nv_bfloat16* __restrict__ dout,
                                  __nv_bfloat16* __restrict__ qr, __nv_bfloat16* __restrict__ kr,
                                  float* __restrict__ delta, float* __restrict__ dq_acc,
                                  const Problem pb, RopeTable rope, int* status) {
  pdl_wait();  // the forward that wrote O (and anything before it) has completed
  const int seq = blockIdx.y;
  int start, len;
  // A sequence whose cu_seqlens bounds are invalid is skipped by all three
  // kernels; the first CTA of its row reports it.
  if (!seq_bounds(pb, seq, start, len, (blockIdx.x == 0 && threadIdx.x == 0) ? status : nullptr))
    return;
  const int t0 = blockIdx.x * bwd::kPreRows;
  if (t0 >= len) return;
  const int H = pb.H;
  const int items = min(bwd::kPreRows, len - t0) * H * 8;
  const int items_all = (items + 255) & ~255;  // every thread runs every round (shuffles)
  for (int w = threadIdx.x; w < items_all; w += 256) {
    const bool valid = w < items;
    const int part = w & 7;
    // A lane past the last item works on item 0 of the block (always inside
    // the sequence) and discards the result, so that every address it forms
    // is valid.
    const int rh = valid ? (w >> 3) : 0;
    const int rr = rh / H, h = rh - rr * H;
    const int pos = t0 + rr;
    const long long pair = static_cast<long long>(start + pos) * H + h;
    float acc = 0.f;
    if (valid) {
      const uint4 o = __ldg(reinterpret_cast<const uint4*>(out + pair * kHD) + part);
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(dout + pair * kHD) + part);
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc = __fmaf_rn(bf16lo_to_f32(ow[u]), bf16lo_to_f32(gw[u]), acc);
        acc = __fmaf_rn(bf16hi_to_f32(ow[u]), bf16hi_to_f32(gw[u]), acc);
      }
      float4* z = reinterpret_cast<float4*>(dq_acc + pair * kHD) + part * 2;
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      // RoPE of one chunk pair of q (parts 0-3) or k (parts 4-7).
      const int c = part & 3;
      const __nv_bfloat16* src = (part < 4 ? q : k) + pair * kHD;
      __nv_bfloat16* dst = (part < 4 ? qr : kr) + pair * kHD;
      const uint4 lo = __ldg(reinterpret_cast<const uint4*>(src) + c);
      const uint4 hi = __ldg(reinterpret_cast<const uint4*>(src) + c + 4);
      const float4* cs = reinterpret_cast<const float4*>(rope.cs + static_cast<long long>(pos) * 32 + 8 * c);
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
      reinterpret_cast<uint4*>(dst)[c] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      reinterpret_cast<uint4*>(dst)[c + 4] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (valid && part == 0) delta[static_cast<long long>(h) * pb.n_tot + start + pos] = acc;
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// 1'. preprocess when q', k' are the caller's (nothing to rotate): a
//     persistent stream over the (row, head) pairs of the packed tensors.
//     Each CTA (kPrepCtasPerSm per SM) takes an even share of the pairs in
//     chunks of at most kPrepPairs.  Thread 0 bulk-copies the O and dO rows
//     of a chunk into one of kPrepStages shared-memory stages, kPrepStages
//     chunks ahead; all threads zero the chunk's dQ' rows, then form D_m from
//     the staged rows with 8 threads per pair and the partial sums and
//     shuffle tree of the kernel above, so that D is bitwise the same.  Rows
//     outside every sequence (a packed batch with gaps, or a sequence with
//     bad bounds) get D and zeroed dQ' rows too; nothing reads them.
// ---------------------------------------------------------------------------
namespace bwd {
constexpr int kPrepPairs = 128;  // pairs per chunk
constexpr int kPrepStages = 2;
constexpr int kPrepCtasPerSm = 3;
constexpr int kPrepRowBytes = kHD * 2;                           // one bf16 row of O or dO
constexpr int kPrepStageBytes = 2 * kPrepPairs * kPrepRowBytes;  // O rows, then dO rows
constexpr int PREP_SMEM_BYTES = kPrepStages * kPrepStageBytes + kPrepStages * 8 + 16;
}  // namespace bwd

__global__ void __launch_bounds__(256, bwd::kPrepCtasPerSm)
    ne_attn_bwd_prep_stream_kernel(const __nv_bfloat16* __restrict__ out,
                                   const __nv_bfloat16* __restrict__ dout,
                                   float* __restrict__ delta, float* __restrict__ dq_acc,
                                   const Problem pb, int* status) {
  using namespace bwd;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPrepStages * kPrepStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kPrepStages);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kPrepStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // This CTA's share of dO into L2 while the forward finishes (dO is an input
  // of the call, which the forward does not write; a prefetch is only a hint).
  if (tid == 0) {
    const long long all = static_cast<long long>(pb.n_tot) * pb.H;
    const long long a = all * blockIdx.x / gridDim.x, e = all * (blockIdx.x + 1) / gridDim.x;
    if (e > a)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                       reinterpret_cast<uint64_t>(dout + a * kHD)),
                   "r"(static_cast<uint32_t>((e - a) * kPrepRowBytes))
                   : "memory");
  }
  pdl_wait();  // the forward that wrote O (and anything before it) has completed
  // Bad cu_seqlens entries are reported here; the main kernel and the
  // postprocess skip those sequences.
  if (pb.cu_seqlens && blockIdx.x == 0) {
    for (int s = tid; s < pb.nseq; s += 256) {
      int a, l;
      seq_bounds(pb, s, a, l, status);
    }
  }
  const int H = pb.H;
  const long long n_pairs = static_cast<long long>(pb.n_tot) * H;
  const long long p0 = n_pairs * blockIdx.x / gridDim.x;
  const int mine = static_cast<int>(n_pairs * (blockIdx.x + 1) / gridDim.x - p0);
  const int n_ch = (mine + kPrepPairs - 1) / kPrepPairs;
  // Chunk j: pairs p0 + first(j) .. p0 + first(j + 1) - 1 (at most kPrepPairs),
  // split as evenly as the count allows (32-bit arithmetic from here on: the
  // pair p0 + t is row m0 + (h0 + t) / H, head (h0 + t) % H).
  const int per = n_ch ? mine / n_ch : 0, extra = n_ch ? mine - per * n_ch : 0;
  auto first = [&](int j) { return j * per + min(j, extra); };
  const long long m0 = p0 / H;
  const int h0 = static_cast<int>(p0 - m0 * H);
  auto issue = [&](int j) {
    const int s = j % kPrepStages;
    const long long b = p0 + first(j);
    const uint32_t bytes = static_cast<uint32_t>(first(j + 1) - first(j)) * kPrepRowBytes;
    uint8_t* st = smem + s * kPrepStageBytes;
    mbar_arrive_expect_tx(&full[s], 2u * bytes);
    bulk_load(st, out + b * kHD, bytes, &full[s]);
    bulk_load(st + kPrepPairs * kPrepRowBytes, dout + b * kHD, bytes, &full[s]);
  };
  int issued = 0;  // thread 0 only
  if (tid == 0)
    for (; issued < n_ch && issued < kPrepStages; ++issued) issue(issued);
  int j = 0;
  for (; j < n_ch; ++j) {
    const int s = j % kPrepStages;
    const int t0 = first(j);
    const long long b = p0 + t0;
    const int np = first(j + 1) - t0;
    // The chunk's dQ' rows (np x 64 fp32), while its O and dO rows land.
    uint4* z = reinterpret_cast<uint4*>(dq_acc + b * kHD);
    for (int i = tid; i < np * (kHD / 4); i += 256) z[i] = make_uint4(0u, 0u, 0u, 0u);
    const bool ok = mbar_wait(&full[s], (j / kPrepStages) & 1, abort_flag, status, 45);
    if (!__syncthreads_and(ok)) break;
    const uint8_t* so = smem + s * kPrepStageBytes;
    const uint8_t* sg = so + kPrepPairs * kPrepRowBytes;
    const int items = np * 8;
    const int items_all = (items + 255) & ~255;  // every thread runs every round (shuffles)
    for (int w = tid; w < items_all; w += 256) {
      const bool valid = w < items;
      const int part = w & 7;
      const int pr = valid ? (w >> 3) : 0;  // a lane past the end reads pair 0, discarded
      const uint4 o = *reinterpret_cast<const uint4*>(so + pr * kPrepRowBytes + part * 16);
      const uint4 g = *reinterpret_cast<const uint4*>(sg + pr * kPrepRowBytes + part * 16);
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc = __fmaf_rn(bf16lo_to_f32(ow[u]), bf16lo_to_f32(gw[u]), acc);
        acc = __fmaf_rn(bf16hi_to_f32(ow[u]), bf16hi_to_f32(gw[u]), acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      if (valid && part == 0) {
        const int t = h0 + t0 + pr;
        const int dm = t / H;
        delta[static_cast<long long>(t - dm * H) * pb.n_tot + m0 + dm] = acc;
      }
    }
    __syncthreads();  // stage s has been read: refill it
    if (tid == 0 && issued < n_ch) issue(issued++);
  }
  if (tid == 0) {
    // After an abort, the loads still in flight land before the CTA exits.
    for (; j < issued; ++j) {
      const long long t0 = clock64();
      while (!mbar_try_wait(&full[j % kPrepStages], (j / kPrepStages) & 1) &&
             clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
      }
    }
  }
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// 2. main kernel: persistent.  A unit is one 128-key tile kt of one (sequence,
//    head); the CTAs (one per SM) walk the units longest first (key tile 0,
//    whose query tiles are the most, for every (sequence, head), then tile 1,
//    ...), dealt in a snake order -- or, for a fixed-length batch, by a
//    schedule packed on the host.  TMEM, barriers and the Q'/dO ring persist
//    across units, so a unit's start (its K', V loads, first S^T/dP^T) overlaps
//    the previous unit's tail (last dQ' drain, dV/dK epilogue) instead of
//    waiting for a new CTA.  Barrier phases count query tiles over all of the
//    CTA's units (ring stages and per-tile hand-offs) or units (K', V).
// ---------------------------------------------------------------------------
namespace bwd {

// One unit: key tile kt of (sequence seq, head h).
struct Unit {
  int seq, h, kt;
  int start, len;  // the sequence's first row in the packed tensors, its length
  int n_it;        // query tiles kt .. n_qt - 1
};

// Unit r of the longest-first order; false for an empty unit (the sequence
// has no such key tile, or a bad cu_seqlens entry).
__device__ __forceinline__ bool get_unit(const BwdParams& p, int r, Unit& u) {
  const int n_sh = p.pb.nseq * p.pb.H;
  const int sh = r % n_sh;
  u.kt = r / n_sh;
  u.seq = sh / p.pb.H;
  u.h = sh % p.pb.H;
  if (!seq_bounds(p.pb, u.seq, u.start, u.len, nullptr)) return false;
  if (u.kt * kBN >= u.len) return false;
  u.n_it = (u.len + kBM - 1) / kBM - u.kt;
  return true;
}

// The first k' >= k whose unit is not empty (its description in u), or -1.
__device__ __forceinline__ int next_unit(const BwdParams& p, int n_units, int c, int G, int k,
                                         Unit& u) {
  for (;; ++k) {
    const int r = dealt_item(p.sched, p.compact, k, c, G, n_units);
    if (r >= n_units) return -1;
    if (get_unit(p, r, u)) return k;
  }
}

}  // namespace bwd

__global__ void __launch_bounds__(512, 1)
    ne_attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDQ,
                       const __grid_constant__ CUtensorMap tmDV,
                       const __grid_constant__ CUtensorMap tmDK, const BwdParams p, int n_tiles) {
  using namespace bwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * B_COUNT + 4);

  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int n_units = n_tiles * p.pb.nseq * p.pb.H;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[B_K_FULL + b], 1);
      mbar_init(&bars[B_K_EMPTY + b], 2);  // one commit from each issuing warp
    }
    mbar_init(&bars[B_V_FULL], 1);
    mbar_init(&bars[B_V_EMPTY], 1);
    mbar_init(&bars[B_EPI_FULL], 256);
    mbar_init(&bars[B_EPI_READ], 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars[B_QDO_FULL + s], 1);
      mbar_init(&bars[B_QDO_EMPTY + s], 1);
    }
    for (int s = 0; s < kRowSlots; ++s) {
      mbar_init(&bars[B_ROW_FULL + s], 128);
      mbar_init(&bars[B_ROW_EMPTY + s], 8);  // one arrival per softmax warp
    }
    mbar_init(&bars[B_S_FULL], 1);
    mbar_init(&bars[B_S_FREE], 256);
    mbar_init(&bars[B_DS_FULL], 256);
    mbar_init(&bars[B_PDS_FREE], 1);
    mbar_init(&bars[B_DQ_FULL], 1);
    mbar_init(&bars[B_DQ_FREE], 128);
    mbar_init(&bars[B_MMA_DONE], 1);
    mbar_init(&bars[B_SDP_DONE], 1);
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
  pdl_wait();  // the preprocess (q', k', D, zeroed dQ') has completed
  pdl_launch_dependents();

  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  uint8_t* sQ = smem + OFF_Q;
  uint8_t* sDO = smem + OFF_DO;
  uint8_t* sDST = smem + OFF_DST;
  uint8_t* sDQ = smem + OFF_DQ;
  float* sLSE = reinterpret_cast<float*>(smem + OFF_LSE);
  float* sDEL = reinterpret_cast<float*>(smem + OFF_DEL);
  // The units of this CTA, in order (the same sequence in every role).
#define NE_FOR_EACH_UNIT(u)                                                                   \
  for (int k_ = 0, r_ = dealt_item(p.sched, p.compact, 0, cta, G, n_units); r_ < n_units;     \
       ++k_, r_ = dealt_item(p.sched, p.compact, k_, cta, G, n_units))                           \
    if (Unit u; get_unit(p, r_, u))

  if (warp == 13 || warp == 15) {
    // ------------------------------- TMA producers: warp 13 Q'/dO, warp 15 K'/V
    regs_decrease<kRegsMma>();
    if (lane == 0 && warp == 13) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      bool ok = true;
      int g = 0;  // query tiles loaded over all units
      int last_issued[kQStages] = {-1, -1, -1};
      NE_FOR_EACH_UNIT(u) {
        if (!ok) break;
        for (int it = 0; it < u.n_it; ++it, ++g) {
          const int s = g % kQStages;
          if (g >= kQStages &&
              !mbar_wait(&bars[B_QDO_EMPTY + s], ((g - kQStages) / kQStages) & 1, abort_flag,
                         p.status, 31)) {
            ok = false;
            break;
          }
          const int qrow = u.start + (u.kt + it) * kBM;
          mbar_arrive_expect_tx(&bars[B_QDO_FULL + s], 2 * kTileBytes);
          tma_load_3d(sQ + s * kTileBytes, &tmQ, &bars[B_QDO_FULL + s], 0, u.h, qrow);
          tma_load_3d(sDO + s * kTileBytes, &tmDO, &bars[B_QDO_FULL + s], 0, u.h, qrow);
          last_issued[s] = g;
        }
      }
      if (*abort_flag) {  // copies in flight land before the CTA exits
        for (int s = 0; s < kQStages; ++s)
          if (last_issued[s] >= 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[B_QDO_FULL + s], (last_issued[s] / kQStages) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
      }
    } else if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int nu = 0;  // units loaded
      int last_k[2] = {-1, -1};
      bool ok = true;
      NE_FOR_EACH_UNIT(u) {
        const int b = nu & 1;
        // K' buffer b last held unit nu - 2: free once both issuing warps'
        // last MMAs reading it (that unit's last S^T; its last dQ') completed.
        // It was released a unit ago, so this load runs a unit ahead.
        if (nu >= 2 &&
            !mbar_wait(&bars[B_K_EMPTY + b], ((nu - 2) >> 1) & 1, abort_flag, p.status, 30)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars[B_K_FULL + b], kTileBytes);
        tma_load_3d(sK + b * kTileBytes, &tmK, &bars[B_K_FULL + b], 0, u.h, u.start + u.kt * kBN);
        last_k[b] = nu;
        // V: the one buffer is free once the previous unit's last dP^T completed.
        if (nu >= 1 && !mbar_wait(&bars[B_V_EMPTY], (nu - 1) & 1, abort_flag, p.status, 29)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars[B_V_FULL], kTileBytes);
        tma_load_3d(sV, &tmV, &bars[B_V_FULL], 0, u.h, u.start + u.kt * kBN);
        ++nu;
      }
      if (!ok || *abort_flag) {  // copies in flight land before the CTA exits
        for (int b = 0; b < 2; ++b)
          if (last_k[b] >= 0) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&bars[B_K_FULL + b], (last_k[b] >> 1) & 1) &&
                   clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
            }
          }
        if (nu >= 1) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&bars[B_V_FULL], (nu - 1) & 1) &&
                 clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
          }
        }
      }
    } else if (warp == 15 && lane == 1) {
      // Tile stores of each unit's dV and scale dK', once the softmax threads
      // have staged them in the dS^T buffer (a thread of its own, so that no
      // softmax warp waits for the stores); the buffer is handed back when
      // the stores have read it.  Partial tiles are written by the softmax
      // threads themselves: only the hand-back is needed.
      tma_prefetch_desc(&tmDV);
      tma_prefetch_desc(&tmDK);
      int nu = 0;
      NE_FOR_EACH_UNIT(u) {
        if (!mbar_wait(&bars[B_EPI_FULL], nu & 1, abort_flag, p.status, 50)) break;
        if ((u.kt + 1) * kBN <= u.len) {
          const int row0 = u.start + u.kt * kBN;
          tma_store_3d(&tmDV, sDST, 0, u.h, row0);
          tma_store_3d(&tmDK, sDST + kTileBytes, 0, u.h, row0);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        mbar_arrive(&bars[B_EPI_READ]);
        ++nu;
      }
      bulk_wait_group0();  // the stores have completed before the kernel ends
    }
  } else if (warp == 12 || warp == 14) {
    // ------------------------------------------------------------ MMA issuers
    // Each issuing warp runs its loop and waits with the whole warp; the
    // elected lane issues each group of MMAs together with the commits that
    // track it.  Descriptors: a K step or a ring stage only adds a constant
    // to the start-address field (16-byte units).
    regs_decrease<kRegsMma>();
    constexpr uint64_t kTileD = kTileBytes >> 4;
    uint64_t* done = &bars[warp == 12 ? B_MMA_DONE : B_SDP_DONE];
    bool ok = true;
    int g = 0;   // query tiles over all units
    int nu = 0;  // units
    if (warp == 14) {
      const uint64_t dKk = make_sdesc_sw128(smem_u32(sK), 16, 1024);    // K' K-major
      const uint64_t dVk = make_sdesc_sw128(smem_u32(sV), 16, 1024);    // V K-major
      const uint64_t dQk0 = make_sdesc_sw128(smem_u32(sQ), 16, 1024);   // Q' K-major
      const uint64_t dOk0 = make_sdesc_sw128(smem_u32(sDO), 16, 1024);  // dO K-major
      // S^T = K' Q'^T and dP^T = V dO^T of every query tile, as soon as Q_n
      // and dO_n have landed and the softmax has read the previous S^T, dP^T.
      NE_FOR_EACH_UNIT(u) {
        if (!ok) break;
        const int b = nu & 1;
        if (!mbar_wait_warp(&bars[B_K_FULL + b], (nu >> 1) & 1, abort_flag, p.status, 32) ||
            !mbar_wait_warp(&bars[B_V_FULL], nu & 1, abort_flag, p.status, 38)) {
          ok = false;
          break;
        }
        for (int it = 0; it < u.n_it; ++it, ++g) {
          const int sn = g % kQStages;
          if (!mbar_wait_warp(&bars[B_QDO_FULL + sn], (g / kQStages) & 1, abort_flag, p.status, 33) ||
              (g >= 1 && !mbar_wait_warp(&bars[B_S_FREE], (g - 1) & 1, abort_flag, p.status, 34))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t dQ = opaque_u64(dQk0) + kTileD * sn, dO = opaque_u64(dOk0) + kTileD * sn;
            const uint64_t dK = opaque_u64(dKk) + kTileD * b, dV = opaque_u64(dVk);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 64 head dims: 32 bytes per step
              umma_bf16_ss(tmem + kColS, dK + 2 * kk, dQ + 2 * kk, kIdescNN, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_ss(tmem + kColDP, dV + 2 * kk, dO + 2 * kk, kIdescNN, kk > 0 ? 1u : 0u);
            umma_commit(&bars[B_S_FULL]);
            if (it == u.n_it - 1) {  // the unit's last readers of V and (here) of K'
              umma_commit(&bars[B_V_EMPTY]);
              umma_commit(&bars[B_K_EMPTY + b]);
            }
          }
          __syncwarp();
        }
        ++nu;
      }
    } else {
      // dV, dK' and dQ' of every query tile, once its softmax is done.
      const uint64_t dKm = make_sdesc_sw128(smem_u32(sK), kTileBytes, 1024);    // K' MN-major
      const uint64_t dQm0 = make_sdesc_sw128(smem_u32(sQ), kTileBytes, 1024);   // Q' MN-major
      const uint64_t dOm0 = make_sdesc_sw128(smem_u32(sDO), kTileBytes, 1024);  // dO MN-major
      const uint64_t dSk = make_sdesc_sw128(smem_u32(sDST), 16, 1024);          // dS^T K-major
      const uint64_t dSm = make_sdesc_sw128(smem_u32(sDST), kTileBytes, 1024);  // as dS, MN-major
      NE_FOR_EACH_UNIT(u) {
        if (!ok) break;
        const int b = nu & 1;
        // K' of this unit (B operand of dQ') has landed.
        if (!mbar_wait_warp(&bars[B_K_FULL + b], (nu >> 1) & 1, abort_flag, p.status, 37)) {
          ok = false;
          break;
        }
        for (int it = 0; it < u.n_it; ++it, ++g) {
          const int s = g % kQStages;
          if (!mbar_wait_warp(&bars[B_DS_FULL], g & 1, abort_flag, p.status, 35)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t dQm = opaque_u64(dQm0) + kTileD * s, dOm = opaque_u64(dOm0) + kTileD * s;
            const uint64_t dS = opaque_u64(dSk);
            // The unit's first tile overwrites dV, dK': the softmax threads
            // read the previous unit's values (their epilogue) before they
            // arrived on DS_FULL for this tile.
            const uint32_t acc0 = it > 0 ? 1u : 0u;
            // dV += P^T dO  (A: P^T in TMEM, 16 queries = 8 packed columns per
            // step; B: dO MN-major, 16 rows = 2048 bytes per step)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ts(tmem + kColDV, tmem + kColPT + 8 * kk, dOm + 128 * kk, kIdescKM,
                           kk > 0 ? 1u : acc0);
            // dK' += dS^T Q'  (A: dS^T K-major, 64-query blocks 16 KiB apart)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_bf16_ss(tmem + kColDK, dS + kTileD * (kk >> 2) + 2 * (kk & 3), dQm + 128 * kk,
                           kIdescKM, kk > 0 ? 1u : acc0);
            // Q_it, dO_it are free: their S^T, dP^T completed before the
            // softmax of the tile began, and dV, dK' are their last readers.
            umma_commit(&bars[B_QDO_EMPTY + s]);
          }
          __syncwarp();
          // dQ'_i = dS K'  (A: dS^T read MN-major, i.e. as dS; B: K' MN-major)
          if (g >= 1 && !mbar_wait_warp(&bars[B_DQ_FREE], (g - 1) & 1, abort_flag, p.status, 36)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t dSq = opaque_u64(dSm), dKq = opaque_u64(dKm) + kTileD * b;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // K = 128 keys: 16 rows = 2048 bytes per step
              umma_bf16_ss(tmem + kColDQ, dSq + 128 * kk, dKq + 128 * kk, kIdescMM,
                           kk > 0 ? 1u : 0u);
            umma_commit(&bars[B_DQ_FULL]);
            umma_commit(&bars[B_PDS_FREE]);
            if (it == u.n_it - 1) umma_commit(&bars[B_K_EMPTY + b]);  // last reader of K'
          }
          __syncwarp();
        }
        ++nu;
      }
    }
    // Drain: every MMA this warp issued completes before TMEM is released.
    if (elect_one()) umma_commit(done);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(done, 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------ row terms and dQ' drain
    regs_decrease<kRegsDrain>();
    const int r = threadIdx.x;  // 0..127: query row of the tile (TMEM lane r)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    // Row terms: a stream over all of the CTA's query tiles, across unit
    // boundaries, kRowSlots - 1 tiles ahead of the drain (so a unit's first
    // tiles are staged during the previous unit).  Cursor: unit ua (index
    // ka, -1 past the end), its tile ita, the CTA's tile number ga.
    Unit ua;
    int ka = next_unit(p, n_units, cta, G, 0, ua);
    int ita = 0, ga = 0;
    // LSE (log2 units) and D of query row r of the cursor's tile; rows past
    // the sequence get LSE = +inf, hence P = 0.  The loads always address a
    // row of the sequence (read-only loads may run ahead of the condition
    // that guards them).
    auto load_rowstats = [&](float& l2, float& dl) {
      const int qpos = (ua.kt + ita) * kBM + r;
      const int qc = qpos < ua.len ? qpos : ua.len - 1;
      const float l = __ldg(p.lse + lse_index(p.pb, ua.h, ua.seq, ua.start, qc));
      const float d = __ldg(p.delta + static_cast<long long>(ua.h) * p.pb.n_tot + ua.start + qc);
      l2 = qpos < ua.len ? l * 1.4426950408889634f : INFINITY;
      dl = qpos < ua.len ? d : 0.f;
    };
    // Stored negated: P = 2^(fma(s, scale log2 e, -LSE)), dS = P (dP - D).
    // The slot last held tile ga - kRowSlots, whose readers have all
    // arrived on its ROW_EMPTY phase (the next phase of that barrier needs
    // this staging first, so the parity cannot alias).
    auto stage_rowstats = [&](float l2, float dl) -> bool {
      const int sl = ga % kRowSlots;
      if (ga >= kRowSlots &&
          !mbar_wait_warp(&bars[B_ROW_EMPTY + sl], ((ga - kRowSlots) / kRowSlots) & 1, abort_flag,
                          p.status, 44))
        return false;
      sLSE[sl * 128 + r] = -l2;
      sDEL[sl * 128 + r] = -dl;
      mbar_arrive(&bars[B_ROW_FULL + sl]);
      ++ga;
      if (++ita == ua.n_it) {
        ita = 0;
        ka = next_unit(p, n_units, cta, G, ka + 1, ua);
      }
      return true;
    };
    float l2, dl;
    for (int j = 0; j < kRowSlots - 1 && ka >= 0; ++j) {  // no waits: slots not yet used
      load_rowstats(l2, dl);
      stage_rowstats(l2, dl);
    }
    int g = 0;  // query tiles over all units
    NE_FOR_EACH_UNIT(u) {
      for (int it = 0; it < u.n_it; ++it) {
        const int gq = g + it;
        const bool ahead = ka >= 0;  // tile gq + kRowSlots - 1 exists: its row terms are next
        if (ahead) load_rowstats(l2, dl);  // loads in flight during the drain
        // dQ'_it: TMEM -> swizzled fp32 staging (columns 0-31 and 32-63) ->
        // two bulk tensor reduce-adds, issued by thread 0.  The four warps
        // meet at named barriers; a warp whose bounded wait gave up carries
        // that into the first barrier's vote, and all four leave together.
        uint32_t v0[32], v1[32];
        bool wok = mbar_wait_warp(&bars[B_DQ_FULL], gq & 1, abort_flag, p.status, 43);
        if (wok) {
          tc_fence_after();
          tmem_ld_x32(tmem + lane_base + kColDQ, v0);
          tmem_ld_x32(tmem + lane_base + kColDQ + 32, v1);
          tmem_ld_wait(v0);
          tmem_ld_wait(v1);
          tc_fence_before();
          mbar_arrive(&bars[B_DQ_FREE]);
        }
        // The staging buffers are free once the previous reductions have read them.
        if (r == 0) bulk_wait_group_read0();
        if (!(ok = named_bar_and(1, 128, ok && wok))) break;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(sDQ + sw128_offset(r, c)) =
              make_uint4(v0[4 * c], v0[4 * c + 1], v0[4 * c + 2], v0[4 * c + 3]);
          *reinterpret_cast<uint4*>(sDQ + kTileBytes + sw128_offset(r, c)) =
              make_uint4(v1[4 * c], v1[4 * c + 1], v1[4 * c + 2], v1[4 * c + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (r == 0) {
          const int qrow = u.start + (u.kt + it) * kBM;
          tma_reduce_add_3d(&tmDQ, sDQ, 0, u.h, qrow);
          tma_reduce_add_3d(&tmDQ, sDQ + kTileBytes, 32, u.h, qrow);
          bulk_commit_group();
        }
        // A failure here is carried into the next tile's vote.
        if (ahead) ok = stage_rowstats(l2, dl);
      }
      // (No exit here: a failure reaches the next tile's vote, or the loops
      // simply end after the CTA's last tile.)
      g += u.n_it;
    }
    // Every reduce-add has completed (not only read its source) before the
    // kernel ends.
    if (r == 0) bulk_wait_group0();
  } else {
    // --------------------------------------------------------- softmax warps
    regs_increase<kRegsSoftmax>();
    const int half = (warp - 4) >> 2;  // query columns 64*half .. 64*half+63
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // key row in tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g = 0;   // query tiles over all units
    int nu = 0;  // units
    NE_FOR_EACH_UNIT(u) {
      if (!ok) break;
      for (int it = 0; it < u.n_it; ++it) {
        const int gq = g + it;
        if (!mbar_wait_warp(&bars[B_S_FULL], gq & 1, abort_flag, p.status, 39)) {
          ok = false;
          break;
        }
        // LSE/D of this query tile are staged in slot gq % kRowSlots.
        const int sl = gq % kRowSlots;
        if (!mbar_wait_warp(&bars[B_ROW_FULL + sl], (gq / kRowSlots) & 1, abort_flag, p.status, 40)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The thread's 64 query columns in two halves of 32, one after the
        // other: each half's S^T and dP^T words come in one TMEM round trip.
        // Holding 32 columns instead of 64 leaves the compiler registers to
        // overlap the exponentials' latency (the accumulator columns are
        // released once the second half is in registers).
        const uint32_t cs = kColS + 64 * half, cd = kColDP + 64 * half;
        const float4* nl4 = reinterpret_cast<const float4*>(sLSE + sl * 128 + 64 * half);
        const float4* nd4 = reinterpret_cast<const float4*>(sDEL + sl * 128 + 64 * half);
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        uint32_t pw[32], dw[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t sv[32], dv[32];
          tmem_ld_x32(tmem + lane_base + cs + 32 * hh, sv);
          tmem_ld_x32(tmem + lane_base + cd + 32 * hh, dv);
          tmem_ld_wait(sv);
          tmem_ld_wait(dv);
          if (hh == 1) {
            tc_fence_before();
            mbar_arrive(&bars[B_S_FREE]);  // S^T/dP^T may be overwritten now
          }
          if (it == 0) {
#pragma unroll
            for (int col = 0; col < 32; ++col)
              if (64 * half + 32 * hh + col < r) sv[col] = 0xff800000u;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 nl = nl4[8 * hh + q], nd = nd4[8 * hh + q];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = 4 * q + 2 * e;
              const uint64_t t = f2_fma(f2_pack(__uint_as_float(sv[col]), __uint_as_float(sv[col + 1])),
                                        sl2x2, e ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y));
              float t0, t1;
              f2_unpack(t, t0, t1);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              const uint64_t dd = f2_add(f2_pack(__uint_as_float(dv[col]), __uint_as_float(dv[col + 1])),
                                         e ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y));
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(p0, p1), dd), d0, d1);
              pw[16 * hh + col / 2] = pack_bf16x2(p0, p1);
              dw[16 * hh + col / 2] = pack_bf16x2(d0, d1);
            }
          }
        }
        // This warp is done with the slot's row terms.
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_ROW_EMPTY + sl]);
        // P^T (TMEM) / dS^T (smem): free once the MMAs of the previous tile are
        // done, and at a unit's first tile once the previous unit's dV/dK tile
        // stores have read the dS^T buffer.
        if (gq >= 1 && !mbar_wait_warp(&bars[B_PDS_FREE], (gq - 1) & 1, abort_flag, p.status, 41)) {
          ok = false;
          break;
        }
        if (it == 0 && nu >= 1 &&
            !mbar_wait_warp(&bars[B_EPI_READ], (nu - 1) & 1, abort_flag, p.status, 49)) {
          ok = false;
          break;
        }
        // P^T row r, queries 64*half .. +63 -> TMEM (32 packed columns); dS^T row
        // r -> smem block `half`, all eight 16-byte chunks.
        tmem_st_x32(tmem + lane_base + kColPT + 32 * half, pw);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8)
          *reinterpret_cast<uint4*>(sDST + half * kTileBytes + sw128_offset(r, k8)) =
              make_uint4(dw[4 * k8], dw[4 * k8 + 1], dw[4 * k8 + 2], dw[4 * k8 + 3]);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_DS_FULL]);
      }
      if (!ok) break;
      // ---- epilogue of the unit: dV (first half), scale dK' (second half),
      // the latter still rotated (the postprocess applies R(n)^T, away from
      // the end of the unit, where table loads would hold up the next unit).
      // (Overlapped by the next unit's S^T/dP^T MMAs; its first dV/dK' MMAs
      // need these TMEM columns only after this thread's next DS_FULL arrival.)
      const int kpos = u.kt * kBN + r;
      const bool full_tile = (u.kt + 1) * kBN <= u.len;
      // dV, dK' are final once the last tile's dV/dK' MMAs have completed; a
      // full tile is staged in the dS^T buffer, free once the last dQ' MMA
      // (its last reader) has completed too.
      const int last = g + u.n_it - 1;
      if (!(ok = full_tile ? mbar_wait_warp(&bars[B_PDS_FREE], last & 1, abort_flag, p.status, 42)
                           : mbar_wait_warp(&bars[B_QDO_EMPTY + last % kQStages],
                                            (last / kQStages) & 1, abort_flag, p.status, 42)))
        break;
      tc_fence_after();
      uint32_t gr[64];
      const uint32_t col = half ? kColDK : kColDV;
      tmem_ld_x32(tmem + lane_base + col, gr);
      tmem_ld_x32(tmem + lane_base + col + 32, gr + 32);
      tmem_ld_wait(gr);
      tmem_ld_wait(gr + 32);
      const float sc = half ? p.scale : 1.f;
      uint4 w[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        w[c] = make_uint4(
            pack_bf16x2(__uint_as_float(gr[8 * c + 0]) * sc, __uint_as_float(gr[8 * c + 1]) * sc),
            pack_bf16x2(__uint_as_float(gr[8 * c + 2]) * sc, __uint_as_float(gr[8 * c + 3]) * sc),
            pack_bf16x2(__uint_as_float(gr[8 * c + 4]) * sc, __uint_as_float(gr[8 * c + 5]) * sc),
            pack_bf16x2(__uint_as_float(gr[8 * c + 6]) * sc, __uint_as_float(gr[8 * c + 7]) * sc));
      if (full_tile) {
        // Row r into the swizzled [128 x 64] bf16 tile `half` of the dS^T
        // buffer; one thread stores both tiles with TMA (whole 128-byte rows,
        // instead of 16-byte pieces of 128 rows per warp instruction).
        uint8_t* tile = sDST + half * kTileBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(tile + sw128_offset(r, c)) = w[c];
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_EPI_FULL]);  // warp 15, lane 1 stores the tiles
      } else {
        // The sequence's last, partial key tile: rows past its end belong to
        // the next sequence (or lie past the tensor), so only rows inside it
        // are written, one row per thread.  The dS^T buffer is not used, but
        // the unit still completes both epilogue phases.
        if (kpos < u.len) {
          const long long orow = (static_cast<long long>(u.start + kpos) * p.pb.H + u.h) * kHD;
          uint4* dst = reinterpret_cast<uint4*>((half ? p.dk : p.dv) + orow);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = w[c];
        }
        mbar_arrive(&bars[B_EPI_FULL]);
      }
      g += u.n_it;
      ++nu;
    }
  }
#undef NE_FOR_EACH_UNIT

  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// 3. postprocess: dq = bf16(scale * R(m)^T dq_acc) (grid layer z = 0) and dk
//    rotated in place (layer z = 1).  Grid (blocks of kPostThreads items,
//    sequences, 2); an item is (row, head, part): part c
//    rotates dims 4c..4c+3 against dims 32+4c..32+4c+3.  Items this small
//    keep a thread under 32 registers, so that a full SM's worth of threads
//    is resident and the grid spans several waves (a small last wave costs
//    little); each warp still reads and writes whole 32-byte sectors.
// ---------------------------------------------------------------------------
constexpr int kPostThreads = 256, kPostParts = 8;

// ---------------------------------------------------------------------------
// dK item of the postprocess (grid layer z = 1): dk = R(n)^T dk in place (the
// main kernel wrote scale dK', still rotated).  Items as for dQ: (row, head,
// part), part c rotates dims 4c..4c+3 against 32+4c..32+4c+3, in fp32 from
// bf16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void dk_rotate_item(__nv_bfloat16* __restrict__ dk, const Problem& pb,
                                               const RopeTable& rope, int start, int len) {
  const int H = pb.H;
  const long long w = static_cast<long long>(blockIdx.x) * kPostThreads + threadIdx.x;
  if (w >= static_cast<long long>(len) * H * kPostParts) return;
  const int part = static_cast<int>(w % kPostParts);
  const int rh = static_cast<int>(w / kPostParts);  // (row, head) pairs fit in 32 bits
  const int pos = rh / H, h = rh - pos * H;
  __nv_bfloat16* row = dk + (static_cast<long long>(start + pos) * H + h) * kHD;
  const uint2 lo = *reinterpret_cast<const uint2*>(row + part * 4);
  const uint2 hi = *reinterpret_cast<const uint2*>(row + 32 + part * 4);
  const float4* cs4 =
      reinterpret_cast<const float4*>(rope.cs + static_cast<long long>(pos) * 32 + part * 4);
  const float4 t0 = __ldg(cs4), t1 = __ldg(cs4 + 1);  // (cos, sin) of dims 4c .. 4c + 3
  const float a[4] = {bf16lo_to_f32(lo.x), bf16hi_to_f32(lo.x), bf16lo_to_f32(lo.y), bf16hi_to_f32(lo.y)};
  const float b[4] = {bf16lo_to_f32(hi.x), bf16hi_to_f32(hi.x), bf16lo_to_f32(hi.y), bf16hi_to_f32(hi.y)};
  const float cz[4] = {t0.x, t0.z, t1.x, t1.z};
  const float sz[4] = {t0.y, t0.w, t1.y, t1.w};
  float go[4], gh[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    go[i] = a[i] * cz[i] + b[i] * sz[i];
    gh[i] = b[i] * cz[i] - a[i] * sz[i];
  }
  *reinterpret_cast<uint2*>(row + part * 4) = make_uint2(pack_bf16x2(go[0], go[1]), pack_bf16x2(go[2], go[3]));
  *reinterpret_cast<uint2*>(row + 32 + part * 4) =
      make_uint2(pack_bf16x2(gh[0], gh[1]), pack_bf16x2(gh[2], gh[3]));
}

__global__ void __launch_bounds__(kPostThreads)
    ne_attn_dq_postprocess_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                                  __nv_bfloat16* __restrict__ dk, const Problem pb, RopeTable rope,
                                  float scale, int rotate_out) {
  pdl_wait();  // the main kernel's dQ' reduce-adds and dK stores have completed
  const int seq = blockIdx.y;
  int start, len;
  if (!seq_bounds(pb, seq, start, len, nullptr)) return;
  if (blockIdx.z == 1) {
    dk_rotate_item(dk, pb, rope, start, len);
    pdl_launch_dependents();
    return;
  }
  const int H = pb.H;
  const long long w = static_cast<long long>(blockIdx.x) * kPostThreads + threadIdx.x;
  if (w >= static_cast<long long>(len) * H * kPostParts) return;
  const int part = static_cast<int>(w % kPostParts);
  const int rh = static_cast<int>(w / kPostParts);  // (row, head) pairs fit in 32 bits
  const int pos = rh / H, h = rh - pos * H;
  const long long row_off = (static_cast<long long>(start + pos) * H + h) * kHD;
  const float4 lo = *reinterpret_cast<const float4*>(dq_acc + row_off + part * 4);
  const float4 hi = *reinterpret_cast<const float4*>(dq_acc + row_off + 32 + part * 4);
  const float a[4] = {lo.x * scale, lo.y * scale, lo.z * scale, lo.w * scale};
  const float b[4] = {hi.x * scale, hi.y * scale, hi.z * scale, hi.w * scale};
  float go[4], gh[4];
  if (!rotate_out) {  // the gradient w.r.t. q' itself
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      go[i] = a[i];
      gh[i] = b[i];
    }
  } else {
    const float4* cs4 =
        reinterpret_cast<const float4*>(rope.cs + static_cast<long long>(pos) * 32 + part * 4);
    const float4 t0 = __ldg(cs4), t1 = __ldg(cs4 + 1);  // (cos, sin) of dims 4c .. 4c + 3
    const float cz[4] = {t0.x, t0.z, t1.x, t1.z};
    const float sz[4] = {t0.y, t0.w, t1.y, t1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      go[i] = a[i] * cz[i] + b[i] * sz[i];
      gh[i] = b[i] * cz[i] - a[i] * sz[i];
    }
  }
  __nv_bfloat16* d = dq + row_off;
  *reinterpret_cast<uint2*>(d + part * 4) = make_uint2(pack_bf16x2(go[0], go[1]), pack_bf16x2(go[2], go[3]));
  *reinterpret_cast<uint2*>(d + 32 + part * 4) =
      make_uint2(pack_bf16x2(gh[0], gh[1]), pack_bf16x2(gh[2], gh[3]));
  pdl_launch_dependents();
}

cudaError_t launch_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmDO, const CUtensorMap& tmDQ, const CUtensorMap& tmDV,
                       const CUtensorMap& tmDK, const BwdParams& p, int n_tiles,
                       cudaStream_t stream, cudaEvent_t ev_pre, cudaEvent_t ev_main) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_attn_bwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bwd::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ne_attn_bwd_prep_stream_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               bwd::PREP_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // One persistent CTA per SM (at most one per unit).
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!sm_count[dev] &&
      (e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long n_units = static_cast<long long>(n_tiles) * p.pb.nseq * p.pb.H;
  const int G = static_cast<int>(n_units < sm_count[dev] ? n_units : sm_count[dev]);
  BwdParams pm = p;
  if (pm.sched && pm.sched_ctas != G) pm.sched = nullptr;  // made for another grid: snake order
  if (p.rotate_in) {
    dim3 pre_grid((n_tiles * kBM + bwd::kPreRows - 1) / bwd::kPreRows, p.pb.nseq);
    e = launch_pdl(ne_attn_bwd_preprocess_kernel, pre_grid, dim3(256), 0, stream, p.q, p.k,
                   p.out, p.dout, p.qr, p.kr, p.delta, p.dq_acc, p.pb, p.rope, p.status);
  } else {
    // kPrepCtasPerSm CTAs per SM, each streaming an even share of the pairs.
    const long long chunks = (static_cast<long long>(p.pb.n_tot) * p.pb.H + bwd::kPrepPairs - 1) /
                             bwd::kPrepPairs;
    const long long slots = static_cast<long long>(bwd::kPrepCtasPerSm) * sm_count[dev];
    const int pg = static_cast<int>(chunks < slots ? (chunks > 0 ? chunks : 1) : slots);
    e = launch_pdl(ne_attn_bwd_prep_stream_kernel, dim3(pg), dim3(256), bwd::PREP_SMEM_BYTES,
                   stream, p.out, p.dout, p.delta, p.dq_acc, p.pb, p.status);
  }
  if (e != cudaSuccess) return e;
  if (ev_pre && (e = cudaEventRecord(ev_pre, stream)) != cudaSuccess) return e;
  e = launch_pdl(ne_attn_bwd_kernel, dim3(G), dim3(bwd::kThreads), bwd::SMEM_BYTES, stream, tmQ,
                 tmK, tmV, tmDO, tmDQ, tmDV, tmDK, pm, n_tiles);
  if (e != cudaSuccess) return e;
  if (ev_main && (e = cudaEventRecord(ev_main, stream)) != cudaSuccess) return e;
  const long long post_items = static_cast<long long>(n_tiles) * kBM * p.pb.H * kPostParts;
  // Layer z = 0: dQ from the accumulator; z = 1: dK rotated in place (not
  // when the gradient w.r.t. k' is asked for: the main kernel wrote it).
  dim3 pgrid(static_cast<unsigned>((post_items + kPostThreads - 1) / kPostThreads), p.pb.nseq,
             p.rotate_out ? 2 : 1);
  return launch_pdl(ne_attn_dq_postprocess_kernel, pgrid, dim3(kPostThreads), 0, stream,
                    static_cast<const float*>(p.dq_acc), p.dq, p.dk, p.pb, p.rope, p.scale,
                    p.rotate_out);
}

}  // namespace ne
