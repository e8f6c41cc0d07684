// ne_debug.cu -- bring-up kernels: each exercises one primitive of the
// attention kernels (TMA swizzled tile load, in-smem RoPE, the three tcgen05
// operand forms) in isolation so that a GPU test can check it against host
// arithmetic.
#include "ne_rope.cuh"
#include "ne_sm100.cuh"

namespace ne {

// TMA-load one tile; optionally rotate it; write it out raw or un-swizzled.
__global__ void __launch_bounds__(128, 1)
    ne_debug_tile_kernel(const __grid_constant__ CUtensorMap tm, int h, int row0, int rotate,
                         int pos0, RopeTable rope, uint8_t* dst_raw, __nv_bfloat16* dst_rows,
                         int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kTileBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kTileBytes + 8);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_3d(smem, &tm, bar, 0, h, row0);
  }
  if (!mbar_wait(bar, 0, abort_flag, status, 20)) return;
  const int r = threadIdx.x;
  if (rotate) {
    RopeRow tab;
    rope_load_row(rope, pos0 + r, tab);
    rope_rotate_row(smem, r, tab);
  }
  __syncthreads();
  if (dst_raw) {
    const uint4* s = reinterpret_cast<const uint4*>(smem);
    uint4* d = reinterpret_cast<uint4*>(dst_raw);
    for (int i = threadIdx.x; i < kTileBytes / 16; i += blockDim.x) d[i] = s[i];
  }
  if (dst_rows) {
    for (int c = 0; c < 8; ++c)
      reinterpret_cast<uint4*>(dst_rows + r * 64)[c] =
          *reinterpret_cast<const uint4*>(smem + sw128_offset(r, c));
  }
}

// Write a row-major [rows, 64] bf16 block into smem as swizzled 128-byte rows.
__device__ void debug_store_rows(uint8_t* tile, const __nv_bfloat16* src, int rows,
                                 int src_stride) {
  for (int i = threadIdx.x; i < rows * 8; i += blockDim.x) {
    const int r = i / 8, c = i % 8;
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, c)) =
        *reinterpret_cast<const uint4*>(src + static_cast<long long>(r) * src_stride + c * 8);
  }
}

__global__ void __launch_bounds__(128, 1)
    ne_debug_umma_kernel(int form, const __nv_bfloat16* a, const __nv_bfloat16* b, float* d,
                         int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;                   // up to 2 tiles
  uint8_t* sB = smem + 2 * kTileBytes;  // 1 tile
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 3 * kTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 3 * kTileBytes + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 3 * kTileBytes + 12);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (form == 0) {
    debug_store_rows(sA, a, 128, 64);
    debug_store_rows(sB, b, 128, 64);
  } else if (form == 1) {
    // a [128 rows, 128 K]: two K blocks of 64 columns, each a [128, 64] tile.
    debug_store_rows(sA, a, 128, 128);
    debug_store_rows(sA + kTileBytes, a + 64, 128, 128);
    debug_store_rows(sB, b, 128, 64);  // b [K=128 rows, N=64]
  } else if (form == 2) {
    // a [K=128 rows, M=128]: two M blocks of 64 columns.
    debug_store_rows(sA, a, 128, 128);
    debug_store_rows(sA + kTileBytes, a + 64, 128, 128);
    debug_store_rows(sB, b, 128, 64);
  } else {
    debug_store_rows(sB, b, 128, 64);  // a goes to TMEM below
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ncols = (form == 0) ? 128 : 64;
  if (form == 3) {
    // Row r of a -> TMEM lane r, columns 128..191 (bf16 pairs packed per column).
    const int row = warp * 32 + lane;
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(a + row * 128);
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t r[32];
      for (int c = 0; c < 32; ++c) r[c] = arow[c0 + c];
      tmem_st_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128 + c0, r);
      tmem_st_wait();
    }
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
    if (form == 0) {
      const uint32_t idesc = make_idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16_ss(tmem, make_sdesc_sw128(aA + kk * 32, 16, 1024),
                     make_sdesc_sw128(aB + kk * 32, 16, 1024), idesc, kk > 0);
    } else if (form == 1) {
      const uint32_t idesc = make_idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16_ss(tmem, make_sdesc_sw128(aA + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024),
                     make_sdesc_sw128(aB + kk * 2048, kTileBytes, 1024), idesc, kk > 0);
    } else if (form == 2) {
      const uint32_t idesc = make_idesc_bf16(128, 64, true, true);
      for (int kk = 0; kk < 8; ++kk)
        umma_bf16_ss(tmem, make_sdesc_sw128(aA + kk * 2048, kTileBytes, 1024),
                     make_sdesc_sw128(aB + kk * 2048, kTileBytes, 1024), idesc, kk > 0);
    } else {
      const uint32_t idesc = make_idesc_bf16(128, 64, false, true);
      for (int kk = 0; kk < 8; ++kk)  // 16 K elements = 8 packed TMEM columns per step
        umma_bf16_ts(tmem, tmem + 128 + kk * 8, make_sdesc_sw128(aB + kk * 2048, kTileBytes, 1024),
                     idesc, kk > 0);
    }
    umma_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait_warp(bar, 0, abort_flag, status, 21);
  tc_fence_after();
  if (ok) {
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
      tmem_ld_wait(r);
      for (int c = 0; c < 32; ++c) d[row * ncols + c0 + c] = __uint_as_float(r[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// A two-stage TMA -> tcgen05 pipeline shaped like the attention kernels' own:
// a producer lane streams 128 x 64 tiles A_i into a ring, an MMA warp
// accumulates D += A_i A_i^T in TMEM and frees each stage with a commit, and
// every wait is bounded -- here by the runtime limit `limit` (cycles).  With
// drop_item >= 0 the producer leaves out the load of that item and its arrive,
// so the MMA warp's wait for it expires.  The kernel must then take the
// attention kernels' abort path: the timeout (site 51) is recorded in the
// status word, every role stops, the copies and MMAs already in flight are
// waited for (bounded), TMEM is released, and the kernel exits normally.  D
// (row-major [128, 128] fp32) is written only when nothing aborted.
__global__ void __launch_bounds__(128, 1)
    ne_debug_pipeline_kernel(const __grid_constant__ CUtensorMap tm, int n_items, int drop_item,
                             long long limit, float* d, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kTileBytes);  // FULL 0-1, EMPTY 2-3, DONE 4
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * kTileBytes + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 2 * kTileBytes + 68);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 5; ++b) mbar_init(&bars[b], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 1 && lane == 0) {
    int last_issued[2] = {-1, -1};
    for (int i = 0; i < n_items; ++i) {
      const int s = i & 1;
      if (i >= 2 && !mbar_wait_limit(&bars[2 + s], ((i - 2) >> 1) & 1, abort_flag, status, 50,
                                     limit))
        break;
      if (i == drop_item) continue;  // the left-out producer arrive
      mbar_arrive_expect_tx(&bars[s], kTileBytes);
      tma_load_3d(smem + s * kTileBytes, &tm, &bars[s], 0, 0, i * kBM);
      last_issued[s] = i;
    }
    // Copies in flight land before the CTA exits (after an abort the consumer
    // may not have waited for them).
    {
      for (int s = 0; s < 2; ++s)
        if (last_issued[s] >= 0) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&bars[s], (last_issued[s] >> 1) & 1) &&
                 clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
          }
        }
    }
  } else if (warp == 2) {
    const uint32_t idesc = make_idesc_bf16(128, 128, false, false);
    for (int i = 0; i < n_items; ++i) {
      const int s = i & 1;
      const bool ok =
          mbar_wait_limit(&bars[s], (i >> 1) & 1, abort_flag, status, 51, limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t dA = make_sdesc_sw128(smem_u32(smem + s * kTileBytes), 16, 1024);
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ss(tmem, dA + 2 * kk, dA + 2 * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[2 + s]);
      }
      __syncwarp();
    }
    // Drain: every MMA issued completes before TMEM is read or released.
    if (elect_one()) umma_commit(&bars[4]);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(&bars[4], 0) && clock64() - t0 < NE_WAIT_LIMIT_CYCLES) {
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!*abort_flag) {
    const int row = warp * 32 + lane;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tmem_ld_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
      tmem_ld_wait(r);
      for (int c = 0; c < 32; ++c) d[row * 128 + c0 + c] = __uint_as_float(r[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

cudaError_t launch_debug_pipeline(const CUtensorMap& tm, int n_items, int drop_item,
                                  long long limit, float* d, int* status, cudaStream_t stream) {
  const int smem = 2 * kTileBytes + 128 + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_debug_pipeline_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ne_debug_pipeline_kernel<<<1, 128, smem, stream>>>(tm, n_items, drop_item, limit, d, status);
  return cudaGetLastError();
}

cudaError_t launch_debug_tile(const CUtensorMap& tm, int h, int row0, int rotate, int pos0,
                              RopeTable rope, void* dst_raw, __nv_bfloat16* dst_rows,
                              int* status, cudaStream_t stream) {
  const int smem = kTileBytes + 64 + 1024;
  ne_debug_tile_kernel<<<1, 128, smem, stream>>>(tm, h, row0, rotate, pos0, rope,
                                                 static_cast<uint8_t*>(dst_raw), dst_rows, status);
  return cudaGetLastError();
}

cudaError_t launch_debug_umma(int form, const __nv_bfloat16* a, const __nv_bfloat16* b, float* d,
                              int* status, cudaStream_t stream) {
  const int smem = 3 * kTileBytes + 64 + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ne_debug_umma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ne_debug_umma_kernel<<<1, 128, smem, stream>>>(form, a, b, d, status);
  return cudaGetLastError();
}

}  // namespace ne
