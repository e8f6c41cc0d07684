/*
 * ne_attn_debug.h -- bring-up entry points of the attention library, used by
 * its GPU tests to check each hardware primitive on its own against plain
 * host arithmetic: the TMA 128-byte-swizzled tile load, the in-smem RoPE of a
 * tile, and the three tcgen05 MMA operand forms the attention kernels use;
 * and, on the host alone, the work schedule of the persistent backward.
 * They follow the conventions of ne_attn.h (device pointers owned by the
 * caller, asynchronous on `stream`, host-side argument checks).  The paper
 * pages have no counterpart: these exist only to test the pieces.
 */
#ifndef NE_ATTN_DEBUG_H
#define NE_ATTN_DEBUG_H

#include "ne_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* TMA-load the 128 x 64 tile at rows row0..row0+127, head h of src
 * ([n_rows, H, 64] bf16; rows past n_rows read as zero) into shared memory
 * with the 128-byte swizzle, and copy the 16384 raw shared-memory bytes to
 * dst_raw (device, 16384 bytes). */
ne_status ne_debug_tma_tile(const ne_bf16* src, int n_rows, int H, int h, int row0,
                            void* dst_raw, void* stream);

/* TMA-load the same tile, apply the kernels' in-smem RoPE to every row r at
 * position pos0 + r with the library's cached table for rope_base, and write
 * the rotated tile un-swizzled to dst ([128, 64] bf16). */
ne_status ne_debug_rope_tile(const ne_bf16* src, int n_rows, int H, int h, int row0, int pos0,
                             float rope_base, ne_bf16* dst, void* stream);

/* One tcgen05 MMA chain (bf16 in, fp32 accumulate in TMEM), operands written
 * to shared memory with the software 128-byte swizzle:
 *   form 0: d[128,128] = a[128,64] . b[128,64]^T       (both K-major)
 *   form 1: d[128,64]  = a[128,128] . b[128,64]        (a K-major; b is
 *                                                     [K=128, N=64], MN-major)
 *   form 2: d[128,64]  = a[128,128]^T . b[128,64]      (a is [K=128, M=128],
 *                                                     MN-major; b as form 1)
 *   form 3: d[128,64]  = a[128,128] . b[128,64]        (a held in TMEM, row m
 *                                                     in lane m, bf16 pairs
 *                                                     packed per column; b as
 *                                                     form 1)
 * a, b: row-major bf16 as written above; d: row-major fp32. */
ne_status ne_debug_umma(int form, const ne_bf16* a, const ne_bf16* b, float* d, void* stream);

/* A two-stage TMA -> tcgen05 pipeline shaped like the attention kernels' own
 * (a producer lane streams the 128 x 64 tiles A_i = rows 128 i .. 128 i + 127
 * of head 0 of src into a ring; an MMA warp accumulates d = sum_i A_i A_i^T in
 * TMEM), whose bounded waits use the runtime limit wait_limit_cycles (1000 ..
 * 2e9) instead of the kernels' fixed one.  drop_item = -1: every item is
 * loaded and d ([128, 128] fp32, device) is written.  drop_item = i: the
 * producer leaves out item i's load and its arrive, so the MMA warp's wait for
 * it expires; the kernel then records NE_ERR_TIMEOUT (device code 0x100 + 51)
 * for ne_attn_get_device_status, waits for its copies and MMAs in flight,
 * releases its TMEM and returns without writing d.  This tests the failure
 * path of the kernels without hanging or faulting the GPU (failure detection:
 * the NanoEuler Show HN page, paragraph 5, on training that can be
 * interrupted and resumed).  Requires 1 <= n_items <= 64 and
 * 128 * n_items <= n_rows. */
ne_status ne_debug_pipeline(const ne_bf16* src, int n_rows, int H, int n_items, int drop_item,
                            long long wait_limit_cycles, float* d, void* stream);

/* The work schedule the fixed-length backward calls give their persistent
 * main kernel (host only, no device needed): its units (one key tile of one
 * sequence and head, longest first) for a batch of nseq sequences of length
 * T with H heads, dealt to G CTAs.  Writes the table -- offsets [G + 1], then
 * every CTA's units in the kernel's index order -- into out (HOST, out_len
 * ints) and returns its length: 0 when the snake order is kept (no table),
 * -1 on a bad argument or a table longer than out_len. */
int ne_debug_schedule(int nseq, int H, int T, int G, int* out, int out_len);

#ifdef __cplusplus
}
#endif

#endif /* NE_ATTN_DEBUG_H */
