/*
 * tkg_debug.h — diagnostic entry points of the tkg library.
 *
 * These are not part of the GEMM path.  They expose, for tests, the pieces
 * the GEMM is built from, so that each can be checked in isolation against
 * the definitions it follows:
 *  - the shared-tile swizzle and its compile-time selection (the 32/64/128-byte
 *    XOR layouts of "ThunderKittens: Simple, Fast, and Adorable AI Kernels",
 *    section "Shared Memory Tiles: Automated Swizzling"),
 *  - the L2-aware tile order ("Block Launch Order and L2 Cache Reuse", Table 3),
 *  - a TMA swizzled load, and a single tensor-core MMA on one tile.
 * Host-only functions need no GPU.  Device pointers are caller-owned.
 */
#ifndef TKG_DEBUG_H_
#define TKG_DEBUG_H_

#include <stdint.h>

#include "tkg.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Host: tile coordinates of linear tile id t under the grouped order with
 * super-groups of `group_m` tile-rows (the same function the kernels run).
 * Returns 0, or -1 if an argument is out of range. */
TKG_API int tkg_debug_tile_coord(int t, int tiles_m, int tiles_n, int group_m, int* tm, int* tn);

/* Host: byte offset after the S-byte swizzle (S in {0, 32, 64, 128}) of byte
 * offset `off` in a tile whose base is aligned to 8*S bytes. */
TKG_API uint32_t tkg_debug_swizzle_offset(uint32_t off, uint32_t s_bytes);

/* Host: the swizzle width (128, 64, 32, or 0) chosen for rows of `row_bytes`. */
TKG_API uint32_t tkg_debug_select_swizzle(uint32_t row_bytes);

/* Host: describe a compiled variant.  kind: 0 bf16, 1 fp8, 2 nvfp4; variant as
 * TKG_OPT_VARIANT (>= 1).  info receives {cta_group, tile_n, stages,
 * epilogue_warps, threads, smem_bytes, tile_m} (tile_m: output-tile rows of a
 * CTA pair).  TKG_ERR_INVALID_ARG if absent. */
TKG_API tkg_status tkg_debug_variant_info(int kind, int variant, int32_t info[7]);

/* Host: the variant id tkg_gemm_<kind> would launch for this shape (after
 * TKG_OPT_VARIANT) on a device of `sm_count` SMs; sm_count <= 0 asks the
 * current device (returns -1 if there is none). */
TKG_API int tkg_debug_pick_variant(int kind, int64_t M, int64_t N, int64_t K, int sm_count);

/* Host: the split-K head plan (TKG_OPT_SPLIT_K) for `tiles` output tiles on a
 * persistent grid of `clusters` clusters with `num_kb` K stages per tile:
 * *split_tiles tail tiles cut into *split_s pieces each (0 and 1: no split).
 * Returns 0, or -1 on a null pointer or negative num_kb. */
TKG_API int tkg_debug_split_plan(int64_t tiles, int64_t clusters, int num_kb, int* split_tiles, int* split_s);

/* Host: work item w of that plan: out = {tile, first K stage, end K stage,
 * piece index or -1 for a whole tile}.  Returns 0, or -1 on invalid input. */
TKG_API int tkg_debug_work_item(int w, int split_tiles, int split_s, int num_kb, int out[4]);

/* Fault injection for the device-timeout path: mode 1 makes the next GEMM's
 * producer skip the copies of its first ring stage, mode 2 makes the next
 * attention launch's producer skip the K copies of its first key tile; the
 * consumer's bounded wait runs out and the kernel reports TKG_ERR_TIMEOUT
 * through tkg_check_status.  No copy is ever in flight for the skipped stage.
 * Mode 0 (default) disables it.  The mode applies to the next launch of that
 * kind only. */
TKG_API tkg_status tkg_debug_set_fault(int mode);

/* Tile-visit count for the scheduler check: the next GEMM launch adds 1 to
 * counts[t] (a device array of at least tiles_m * tiles_n zeroed words,
 * caller-owned) each time a CTA (pair) stores output tile t, t being the
 * linear tile id before the grouped reordering.  Every schedule must leave
 * every count at exactly 1.  NULL disables; applies to the next launch only. */
TKG_API tkg_status tkg_debug_set_visit_counter(unsigned int* counts);

/* Device: TMA-load a [64 rows][S bytes] uint8 tile (row pitch S bytes) from
 * `src` with the S-byte swizzle (S in {32, 64, 128}) and copy the raw shared
 * memory image (64*S bytes) to `dst`.  Synchronous on `stream`. */
TKG_API tkg_status tkg_debug_tma_swizzle_probe(int s_bytes, const void* src, void* dst, void* stream);

/* Device: one CTA computes D[128][n] (fp32) = sum over `ksteps` tensor-core
 * MMAs of A·Bᵀ on a single tile.  a_tile: [128][128] bytes, b_tile: [n][128]
 * bytes (K-major rows; bf16 = 64 elements, e4m3 = 128, packed e2m1 = 256 per
 * row); each MMA consumes the next 32 bytes of every row.  kind: 0 bf16,
 * 1 e4m3, 2 nvfp4 block-scaled (scale_vec 4X, e4m3 scales).  For kind 2,
 * sfa_words / sfb_words are the 32-bit contents of 8 tensor-memory columns
 * for each of the 128 lanes ([128][8], lane-major) of the A and B scale
 * regions, and sf_cols[2*i], sf_cols[2*i+1] (each 0..7) select the column of
 * each region used by MMA i.  n in {64, 128, 192, 256}, ksteps in 1..4.
 * a_tile, b_tile, sfa_words, sfb_words and d_out are device pointers (the
 * scale arrays may be NULL for kinds 0 and 1); sf_cols is a host array of
 * 2*ksteps entries (may be NULL for kinds 0 and 1).  Synchronous on `stream`. */
TKG_API tkg_status tkg_debug_mma_probe(int kind, int n, int ksteps, const void* a_tile, const void* b_tile,
                               const uint32_t* sfa_words, const uint32_t* sfb_words, const int32_t* sf_cols,
                               float* d_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TKG_DEBUG_H_ */
