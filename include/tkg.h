/*
 * tkg.h — C ABI of the GB300 (sm_103a) dense tiled tensor-core GEMM.
 *
 *     C = A · Bᵀ        A: [M, K] row-major, B: [N, K] row-major, C: [M, N] row-major bf16
 *
 * The operation is the tile contraction the ThunderKittens paper calls
 * mma_ABt ("att += Q @ K^T" — paper summary "ThunderKittens: Simple, Fast, and
 * Adorable AI Kernels", section "PyTorch-Like Operations on Tiles"), applied to
 * whole matrices the way its GEMM kernel does (same page, "Integration: How the
 * Three Levels Compose", App. B.1 walk-through): bf16 operands, fp32
 * accumulation ("Warp-Level: Tile Operations"), output written back in bf16.
 * The FP8 and NVFP4 variants are the 8-bit and block-scaled 4-bit GEMMs of the
 * Rubin article ("ThunderKittens reaches 22.4 PFLOPS on NVIDIA Rubin", NVFP4
 * paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All matrix pointers are DEVICE pointers, owned by the caller, and must
 *    stay valid until the work queued on `stream` has finished.  The library
 *    never frees or retains them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every GEMM is asynchronous: the call validates, queues one
 *    kernel launch and returns; it never synchronises.
 *  - Accumulation is fp32.  The output is rounded to bf16 with
 *    round-to-nearest-even.  There is no alpha/beta and no accumulate-into-C;
 *    C is overwritten.  C must not overlap A, B or the scales: tiles of C are
 *    stored while other tiles still read the operands.
 *  - M and N are arbitrary (>= 1).  Tiles that run past M, N or K are handled
 *    by the hardware copy engine (zero fill on load, clipping on store), which
 *    is exact for a sum.
 *  - Errors detected before launch are returned and nothing is queued.  Errors
 *    detected on the device (a pipeline wait that exceeded its time limit) are
 *    recorded in a device status word and reported by tkg_check_status().
 *  - The library holds, per device, a small tensor-map cache on the host, a
 *    4-byte status word in a static device variable, stream-ordered scratch
 *    for the NVFP4 scale re-layout (tkg_gemm_nvfp4) and, per stream that ran a
 *    split-K launch (TKG_OPT_SPLIT_K), a 128x256-fp32-per-SM workspace;
 *    tkg_shutdown() releases the host cache and the workspaces.  There is no
 *    CPU fallback: on a device that is not
 *    compute capability 10.3 every GEMM returns TKG_ERR_UNSUPPORTED_DEVICE.
 *  - Entry points are thread-safe.  Calls on different streams may overlap.
 */
#ifndef TKG_H_
#define TKG_H_

#include <stdint.h>

#if defined(__GNUC__)
#define TKG_API __attribute__((visibility("default")))
#else
#define TKG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tkg_status {
    TKG_OK = 0,
    TKG_ERR_INVALID_ARG = 1,        /* a size or pointer argument is out of range */
    TKG_ERR_MISALIGNED = 2,         /* a matrix base pointer is not 16-byte aligned */
    TKG_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not an sm_103 (GB300-class) GPU */
    TKG_ERR_CUDA = 4,               /* a CUDA runtime / driver call failed */
    TKG_ERR_TIMEOUT = 5,            /* a device pipeline wait ran out (see tkg_check_status) */
    TKG_ERR_INTERNAL = 6
} tkg_status;

/* Scale operands.  All pointers are DEVICE pointers, caller-owned.
 *  - FP8:   a_scale / b_scale point to one fp32 each: the dequantisation scale
 *           of A and of B (value = e4m3(code) * scale).  Block-scale pointers
 *           must be NULL.
 *  - NVFP4: a_scale / b_scale point to the fp32 per-tensor scales g_A, g_B;
 *           a_block_scale is e4m3 [M][K/16] row-major (one scale per 16
 *           consecutive K elements of a row of A), b_block_scale is e4m3
 *           [N][K/16] row-major.
 *  - bf16:  pass NULL for the whole struct.
 * The epilogue applies the per-tensor scales as  bf16((acc * a_scale) * b_scale). */
typedef struct tkg_scales {
    const float* a_scale;
    const float* b_scale;
    const uint8_t* a_block_scale;
    const uint8_t* b_block_scale;
} tkg_scales;

/* bf16 GEMM.  A: bf16 [M][K], B: bf16 [N][K], C: bf16 [M][N].
 * Requirements: M, N, K >= 1, each <= 2^31-1; K % 8 == 0 (16-byte row pitch);
 * A, B, C 16-byte aligned.  scales must be NULL.
 * Returns TKG_OK once the kernel is queued. */
TKG_API tkg_status tkg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                         const tkg_scales* scales, void* stream);

/* FP8 GEMM.  A: e4m3 bytes [M][K], B: e4m3 bytes [N][K], C: bf16 [M][N].
 * C = bf16((sum_k e4m3(A[m][k]) * e4m3(B[n][k])) * a_scale * b_scale).
 * Requirements: as bf16 but K % 16 == 0; scales, scales->a_scale and
 * scales->b_scale non-NULL (4-byte aligned device floats). */
TKG_API tkg_status tkg_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                        const tkg_scales* scales, void* stream);

/* NVFP4 block-scaled GEMM.  A: packed e2m1 [M][K/2] bytes, element 2j in the
 * low nibble of byte j; B: packed e2m1 [N][K/2]; C: bf16 [M][N].
 * C = bf16((sum_k (e2m1(A[m][k]) * e4m3(SFA[m][k/16])) *
 *                  (e2m1(B[n][k]) * e4m3(SFB[n][k/16]))) * g_A * g_B).
 * Requirements: as bf16 but K % 32 == 0; all four scale pointers non-NULL;
 * block-scale arrays 16-byte aligned. */
TKG_API tkg_status tkg_gemm_nvfp4(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                          const tkg_scales* scales, void* stream);

/* NVFP4 GEMM that allocates no memory.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory during a
 * call (for example a caller whose device memory belongs to another
 * framework's allocator, one held to a fixed device-memory budget, or one that
 * must not let a call allocate and synchronise in the middle of its own work),
 * because tkg_gemm_nvfp4 takes the scratch for its on-device re-layout of the
 * block scales from a stream-ordered memory pool and may make a per-stream
 * split-K workspace.  Same operation, arguments and layouts as
 * tkg_gemm_nvfp4, planned and launched by the same code, with two
 * differences: the scratch is a fixed array, and the split-K head is never
 * used.  The result is within the NVFP4 tolerance of tkg_gemm_nvfp4's (for
 * shapes where that one runs a split-K head the fp32 summation order differs,
 * so the two need not be bit-identical).  TKG_OPT_SCHEDULE,
 * TKG_OPT_LAUNCH_OVERLAP, TKG_OPT_GROUP_M and TKG_OPT_MAX_CTAS apply as usual.
 *  - Scratch: a fixed device array of TKG_NVFP4_NOALLOC_SCRATCH_BYTES inside
 *    the library, held by every device that loads the library until the
 *    process exits.  A call needs (Ta * 2 + Tn * 2) * ceil(K/256) * 2048
 *    bytes, Ta = ceil(M/256) and Tn = ceil(N/256) being the 256-row and
 *    256-column tile counts of the NVFP4 kernel (its only variant); the limit
 *    fits M = N = K = 16384 exactly.  Larger problems are rejected with
 *    TKG_ERR_INVALID_ARG before any GPU work.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array and each call overwrites the part it uses,
 *    so calls whose GPU work overlaps (e.g. on two streams) race and give
 *    wrong results; order them on one stream or with events.
 *  - It never calls cudaMalloc, cudaFree or any other allocating routine, and
 *    encodes its tensor maps on the stack (no host-side cache entry). */
#define TKG_NVFP4_NOALLOC_SCRATCH_BYTES (32u << 20)
TKG_API tkg_status tkg_gemm_nvfp4_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* C,
                                          const tkg_scales* scales, void* stream);

/* On-device input encoders: fp32 data -> the operands of tkg_gemm_fp8 and
 * tkg_gemm_nvfp4 (the 8-bit and block-scaled 4-bit formats of "ThunderKittens
 * reaches 22.4 PFLOPS on NVIDIA Rubin", NVFP4 and FP8 paragraphs; the pages
 * give the formats, the scale recipe is this library's reading):
 *   FP8:   amax = max|x| over the tensor, q = e4m3(x * (448 / amax)),
 *          *dequant_scale = amax / 448 (1 and q = 0 for an all-zero tensor);
 *          pass q and the scale to tkg_gemm_fp8 as an operand and its scale.
 *   NVFP4: g = amax / (6 * 448); for every row and 16 consecutive elements,
 *          b = max|x| over the block, sb = e4m3(b / (6 g)),
 *          q = e2m1(x / (e4m3(sb) * g)) (q = 0 when that divisor is 0);
 *          q packed two per byte (element 2j in the low nibble of byte j),
 *          block scales [rows][cols/16] e4m3, *global_scale = g; pass them to
 *          tkg_gemm_nvfp4 as an operand, its block scales and its scale.
 * Every multiply and divide is one fp32 IEEE operation; e4m3 / e2m1 rounding
 * is to nearest, ties to even, saturating at 448 / 6, keeping the sign.
 * x: fp32 [rows][cols] row-major; cols % 16 == 0; x and q 16-byte aligned,
 * the scale 4-byte aligned; all device pointers, caller-owned.  The scale
 * output doubles as the amax accumulator while the call runs.  Asynchronous
 * on `stream`: four stream-ordered operations (a 4-byte memset and three
 * kernels), no allocation.  Returns TKG_ERR_INVALID_ARG / TKG_ERR_MISALIGNED
 * before any GPU work for bad arguments. */
TKG_API tkg_status tkg_quantize_fp8(int64_t rows, int64_t cols, const float* x, uint8_t* q, float* dequant_scale,
                                    void* stream);
TKG_API tkg_status tkg_quantize_nvfp4(int64_t rows, int64_t cols, const float* x, uint8_t* q_packed,
                                      uint8_t* block_scales, float* global_scale, void* stream);

/* Non-causal attention forward (the attention example of "ThunderKittens:
 * Simple, Fast, and Adorable AI Kernels", "The Four Functions: Load, Compute,
 * Store, Finish", and the attention prefill of the ThunderKittens DSL page):
 * for every batch b < B and head h < H,
 *   O[b,h] = softmax(Q[b,h] · K[b,h]ᵀ / sqrt(D)) · V[b,h],
 *   lse[b,h,i] = ln Σ_j exp(Q[b,h,i]·K[b,h,j] / sqrt(D))   (if lse != NULL).
 * Q: bf16 [B][H][Nq][D], K and V: bf16 [B][H][Nkv][D], O: bf16 [B][H][Nq][D],
 * all contiguous row-major, 16-byte aligned device pointers; lse: fp32
 * [B][H][Nq], 4-byte aligned, or NULL.  D = 64 or 128; Nq, Nkv >= 1 (any
 * length); B * H <= 65535.  Scores, softmax statistics and the P·V
 * accumulation are fp32; the probabilities enter P·V rounded to bf16; O is
 * rounded to bf16 once.  Buffers are caller-owned; the call allocates nothing
 * and is asynchronous on `stream` (one kernel; with TKG_OPT_LAUNCH_OVERLAP on,
 * a programmatic dependent of the previous kernel).  Bad arguments return
 * TKG_ERR_INVALID_ARG / TKG_ERR_MISALIGNED before any GPU work; device-side
 * wait timeouts surface through tkg_check_status. */
TKG_API tkg_status tkg_attention_fwd(int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, const void* Q,
                                     const void* K, const void* V, void* O, float* lse, void* stream);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns TKG_ERR_TIMEOUT if any kernel since the last check
 * abandoned a pipeline wait (its output is then undefined), TKG_ERR_CUDA if the
 * stream reported an error, else TKG_OK. */
TKG_API tkg_status tkg_check_status(void* stream);

/* Static, never-NULL description of a status code. */
TKG_API const char* tkg_status_string(tkg_status status);

/* Releases host-side caches (tensor maps, per-device launch data) and the
 * library's split-K workspaces (waiting for device work still using them).
 * Device memory owned by the caller is untouched.  Safe to call more than
 * once; the next GEMM call re-initialises. */
TKG_API void tkg_shutdown(void);

/* Tunables (process-wide).  Values persist until changed; 0 restores the
 * default.  Returns TKG_ERR_INVALID_ARG for an unknown key or bad value.
 *  TKG_OPT_TIMEOUT_NS  limit for any single pipeline wait on the device (default 2 s)
 *  TKG_OPT_GROUP_M     super-group height in output tiles for the L2-aware
 *                      tile order (default 16: the {G, N, M/G} order of
 *                      "Block Launch Order and L2 Cache Reuse", Table 3,
 *                      where the paper takes G = 8; 16 reads the least
 *                      from HBM on GB300 with 256-row pair tiles)
 *  TKG_OPT_VARIANT     force a kernel variant: 0 = the default (14 for
 *                      NVFP4; for bf16 and FP8 15 when K >= 2048 and the
 *                      256x512 tiles fill at least four rounds of the
 *                      device's CTA pairs, else 2); 2 = 2-SM (CTA pair)
 *                      256x256 tiles, two tensor-memory accumulators (bf16
 *                      and FP8); 14 = 2-SM 256x256 tiles, one accumulator,
 *                      the block scales brought into shared memory by the
 *                      ring's TMA and copied into tensor memory
 *                      (tcgen05.cp) by four issuing threads (NVFP4);
 *                      15 = 2-SM 256x512 tiles, two
 *                      N = 256 MMAs per K step into all 512 tensor-memory
 *                      columns, the second reusing A from the tensor
 *                      core's collector buffer, eight epilogue warps
 *                      (bf16 and FP8; no split-K head).  A variant
 *                      the kind lacks falls back to the default.
 *  TKG_OPT_MAX_CTAS    cap the persistent grid size (0 = all SMs)
 *  TKG_OPT_LAUNCH_OVERLAP
 *                      TKG_OVERLAP_ON (default): GEMMs are launched as
 *                      programmatic dependents of the previous kernel on the
 *                      stream, so their CTAs set up shared and tensor memory
 *                      on SMs the previous kernel has left while it finishes;
 *                      each CTA still waits for that kernel to complete (and
 *                      its writes to be visible) before it reads A, B or the
 *                      scales or writes C, so stream order is kept.
 *                      TKG_OVERLAP_OFF: plain stream-ordered launches.
 *  TKG_OPT_SCHEDULE    how CTA pairs get output tiles ("Persistent Grid
 *                      Launch", Table 2; Cluster Launch Control):
 *                      TKG_SCHEDULE_STATIC (default) = persistent grid, one
 *                      CTA (pair) per SM, pair c takes tiles c, c + pairs,
 *                      ... in the grouped order;
 *                      TKG_SCHEDULE_DYNAMIC = one cluster per tile is
 *                      launched and running clusters cancel the launch of
 *                      clusters that have not started and take their tiles;
 *                      TKG_SCHEDULE_SINGLE = one cluster per tile, each
 *                      computes its own tile only (non-persistent launch).
 *  TKG_OPT_SPLIT_K     TKG_SPLIT_ON (default): in the static schedule, when
 *                      the persistent grid's last round of tiles would be
 *                      at most half full, those tiles are cut along K into
 *                      S = min(CTA pairs / tail tiles, 4) pieces of at
 *                      least 16 K stages each (bf16: 1024 K elements; a
 *                      grid of one round needs tiles of 48 K stages) that
 *                      run first.  The pieces of a tile share its
 *                      reduction: each writes the fp32 partials of the
 *                      column chunks the others own to a per-stream
 *                      workspace (one fp32 128x256 block per SM, created on
 *                      the stream's first split launch, never while the
 *                      stream is being captured: such launches run
 *                      unsplit), waits (bounded) for the other pieces, and
 *                      adds the partials of its own chunks in piece order,
 *                      so results do not depend on timing.  The pieces are
 *                      the first work items of distinct, co-resident CTA
 *                      pairs.  Not used with the 256x512 tile (variant
 *                      13).  TKG_SPLIT_OFF: whole tiles only.  After a launch reports TKG_ERR_TIMEOUT,
 *                      tkg_check_status frees the workspaces (they are made
 *                      afresh on next use).
 *  TKG_OPT_K_ORDER     TKG_K_ORDER_SERPENTINE (default): each CTA (pair)
 *                      walks the K blocks of its odd-numbered work items
 *                      from the last one down, so that a round of tiles
 *                      starts on the ends of the operand panels the
 *                      previous round read last, which are still in L2;
 *                      TKG_K_ORDER_FORWARD: every item from K block 0 up.
 *                      Only the fp32 summation order changes. */
typedef enum tkg_option {
    TKG_OPT_TIMEOUT_NS = 1,
    TKG_OPT_GROUP_M = 2,
    TKG_OPT_VARIANT = 3,
    TKG_OPT_MAX_CTAS = 4,
    TKG_OPT_LAUNCH_OVERLAP = 5,
    TKG_OPT_SCHEDULE = 6,
    TKG_OPT_SPLIT_K = 7,
    TKG_OPT_K_ORDER = 8
} tkg_option;

/* Values of TKG_OPT_LAUNCH_OVERLAP and TKG_OPT_SCHEDULE. */
#define TKG_OVERLAP_ON 1
#define TKG_OVERLAP_OFF 2
#define TKG_SCHEDULE_STATIC 1
#define TKG_SCHEDULE_DYNAMIC 2
#define TKG_SCHEDULE_SINGLE 3
#define TKG_SPLIT_ON 1
#define TKG_SPLIT_OFF 2
#define TKG_K_ORDER_SERPENTINE 1
#define TKG_K_ORDER_FORWARD 2
TKG_API tkg_status tkg_set_option(tkg_option key, int64_t value);
TKG_API int64_t tkg_get_option(tkg_option key);

#ifdef __cplusplus
}
#endif

#endif /* TKG_H_ */
