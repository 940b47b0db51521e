/*
 * gemm_gb300.h -- C ABI of the GB300 (sm_103a) tcgen05 GEMM library.
 *
 * The library computes, for fp16 or bf16 inputs with fp32 accumulation,
 *
 *     D = alpha * A * B + beta * C
 *
 * The product is the tensor-core operation D = A.B + C that the pages build
 * on ("Tensor Cores, layouts, and swizzling", opening section; "06 Blackwell
 * Tensor Core - tcgen05 MMA", "Overview" and the K-step walk-through: the
 * first K step writes the accumulator, later steps add to it). alpha and
 * beta follow BLAS: beta == 0 never reads C.
 *
 * Operand layouts ("LBO, SBO and SWZ for a tcgen05 tile", section 1:
 * K-major and MN-major operands):
 *   A is logical M x K.   GEMM_K_MAJOR: A[m*lda + k]  GEMM_MN_MAJOR: A[k*lda + m]
 *   B is logical K x N.   GEMM_K_MAJOR: B[n*ldb + k]  GEMM_MN_MAJOR: B[k*ldb + n]
 *   C and D are row-major M x N: C[m*ldc + n], D[m*ldd + n]; C has D's type.
 *
 * Ownership: every pointer is a device pointer owned by the caller; the
 * library allocates no device memory on any call. Calls are asynchronous
 * on `stream` (a cudaStream_t; NULL is the legacy default stream). A call
 * that fails validation returns its error at once and enqueues nothing.
 *
 * Requirements (TMA rules, "Tensor Cores, layouts, and swizzling", TMA
 * section: global strides are multiples of 16 bytes and below 2^40):
 *   - A, B, C, D 16-byte aligned; lda, ldb multiples of 8 elements; ldc and
 *     ldd multiples of 16 bytes of the output type;
 *   - M, N, K >= 0, each below 2^31; leading dimensions at least the
 *     stored row length;
 *   - M == 0 or N == 0: nothing to do (GEMM_OK). K == 0: D = beta * C.
 *   - C == D (in place) is allowed; C may be NULL when beta == 0.
 * Violations return GEMM_ERR_INVALID_ARG or GEMM_ERR_ALIGNMENT.
 *
 * Device-side errors: every wait inside the kernels is bounded. A wait that
 * runs out records a code in a device status word and the kernel returns
 * early; gemm_last_device_status() reads (and clears) that word.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                  /* cudaStream_t is struct CUstream_st* */
typedef struct CUstream_st *gemm_stream_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* bad size, pointer, enum or option */
    GEMM_ERR_ALIGNMENT = 2,          /* pointer or leading dimension breaks a TMA rule */
    GEMM_ERR_UNSUPPORTED = 3,        /* valid request no compiled kernel variant implements */
    GEMM_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed */
    GEMM_ERR_TIMEOUT = 5             /* a bounded device wait ran out */
} gemm_status_t;

typedef enum { GEMM_K_MAJOR = 0, GEMM_MN_MAJOR = 1 } gemm_major_t;

typedef enum { GEMM_OUT_F32 = 0, GEMM_OUT_BF16 = 1, GEMM_OUT_F16 = 2 } gemm_out_t;

/* Shared-memory swizzle of an operand tile ("Swizzling explained properly",
 * "32B, 64B and 128B swizzles"; raw descriptor codes on the LBO/SBO page,
 * section 4). GEMM_SWIZZLE_AUTO lets the library choose (SW128);
 * GEMM_SWIZZLE_NONE stores plain 8-row x 16-byte core matrices (descriptor
 * code 0, LBO and SBO alone define the layout). GEMM_SWIZZLE_128B_ATOM32 is
 * the page's "128-byte mode with 32-byte atomicity" (descriptor code 1):
 * 128-byte rows whose 32-byte units are XORed with the row index mod 4
 * (Swizzle<2,5,2>, written by TMA's 128B_ATOM_32B mode), read as an MN-major
 * operand with K rows in bands of 4. It is the layout of MN-major TF32
 * operands (gemm_ex in_type 2, the default there); 16- and 8-bit operands
 * refuse it with GEMM_ERR_UNSUPPORTED, because kind::f16 and kind::f8f6f4
 * read such operands as zeros on GB300 (measured). */
typedef enum {
    GEMM_SWIZZLE_AUTO = 0,
    GEMM_SWIZZLE_32B = 1,
    GEMM_SWIZZLE_64B = 2,
    GEMM_SWIZZLE_128B = 3,
    GEMM_SWIZZLE_NONE = 4,
    GEMM_SWIZZLE_128B_ATOM32 = 5
} gemm_swizzle_t;

/*
 * Optional tuning/testing knobs (pass NULL for defaults). Every field 0
 * means "library default".
 *   cta_group     1: one CTA per 128-row tile (tcgen05.mma.cta_group::1);
 *                 2: CTA pairs own 256-row tiles (cta_group::2).
 *   tile_m        accumulator rows per CTA: 128, or 64 (cta_group::1 only:
 *                 tcgen05.mma M = 64 with the TMEM accumulator in Layout F,
 *                 "06 Blackwell Tensor Core - tcgen05 MMA", cta_group::1
 *                 M = 64; default for M <= 64 with 16-bit operands), or 32
 *                 (the weight-stationary tcgen05.mma.ws with M = 32; 16-bit
 *                 operands, single problems, tile_n 256), or 256
 *                 (cta_group::1 only: two M = 128 MMAs per K slice share
 *                 each B slice, their accumulators filling the 512 TMEM
 *                 columns; 16-bit operands, single problems, tile_n 256 or
 *                 224; the epilogue of a tile does not overlap the next
 *                 tile's MMAs; by default 256-wide ones run in pairs of CTAs
 *                 that share B, see multicast_b, and the library takes 224
 *                 where that needs fewer rounds of the grid).
 *   tile_n        MMA N per tile: 64, 128 or 256 (cta_group::2: 128 or 256;
 *                 tile_m 256: 224 or 256).
 *   block_k       K elements per pipeline stage: 32, 64 or 128 where built.
 *   swizzle_a/b   operand swizzle (gemm_swizzle_t).
 *   epilogue_swizzle  1 (default) stages output tiles in SW128 layout;
 *                 -1 stages them unswizzled (bank-conflict ablation).
 *   max_ctas      cap on resident CTAs of the persistent grid.
 *   group_m       tile-raster group height in tiles (L2 reuse).
 *   timeout_ms    bound on each device wait (default 2000 ms).
 *   flags         tuning switches. CTA pairs signal stage and accumulator
 *                 releases to both CTAs with one multicast tcgen05.commit;
 *                 bit 0 instead forwards them from the even CTA with remote
 *                 mbarrier arrives (ablation), bit 1 makes every wait
 *                 acquire at cluster scope (ablation). Bit 2 starts each
 *                 tile's K loop at a per-CTA offset so that CTAs sharing an
 *                 operand panel read different parts of it at a time; with
 *                 flags 0 the library sets it for single problems of at most
 *                 one wave of tiles and at least 16 K blocks (HBM-bound
 *                 shapes such as 16384 x 128 x 8192).
 *                 Bit 3 gives the operand loads an L2 evict_last policy and
 *                 the C loads and D stores evict_first (ablation; no
 *                 measured effect at 4096^3 or 8192^3). Bit 4 (single
 *                 problems with 128-row tiles) reads C from global memory
 *                 straight into the epilogue's registers instead of staging
 *                 it in shared memory by TMA (ablation: 1 % slower at 8192^3).
 *                 Bit 5 splits each stage's loads between two producer
 *                 warps, one for the A boxes (and A scale atoms), one for
 *                 the B boxes (and B scale atoms); NVFP4 kernels, which have
 *                 no room for the second warp, ignore it (ablation: no
 *                 measured effect, the loads are bound by L2 delivery, not
 *                 by the issuing thread). Bit 6 (single problems, 128- and
 *                 256-row tiles) writes D from the epilogue's registers with
 *                 16-byte stores, and reads C into them, instead of staging
 *                 chunks in shared memory for TMA (ablation: equal or up to
 *                 5 % slower at 4096^3 and 8192^3).
 *   stats         diagnostics: NULL, or device memory of 16 uint64 per CTA
 *                 of the grid (at least 16 * number of SMs), where each CTA
 *                 writes cycles its roles spent waiting (slots 0-1 producer,
 *                 2-4 and 8-9 MMA issuer, 5-7 and 10-12 first epilogue warp:
 *                 10-11 stream-K flag waits and partial-sum gathers, 12 the
 *                 cycles after its last accumulator became ready; 13 the
 *                 scale copier of the block-scaled kinds, 14 the MMA issuer
 *                 waiting for a stage's scales).
 *   stream_k      K-split scheduling of single (not grouped) problems with
 *                 128-row tiles, so that a last, partly filled wave of tiles
 *                 does not leave SMs idle: the tiles of whole waves run one
 *                 per cluster as usual, and the K blocks of the remaining
 *                 tiles (the ragged wave plus one full wave, or every tile
 *                 when there are fewer tiles than two waves) are divided
 *                 evenly among all clusters. A cluster that holds the first
 *                 K block of a split tile adds the others' fp32 partial sums
 *                 (left in `workspace`) and writes the tile; the result
 *                 differs from the unsplit one only by summation order.
 *                 The pages have no counterpart; it is a scheduling service
 *                 of this library.
 *                   0 (default) auto: split when `workspace` is given and a
 *                     ragged last wave follows 2 to 7 full waves;
 *                  -1 never; 1 always the split above; 2 split every tile;
 *                   3 split only the tiles of the ragged last wave.
 *                 A split needs at least as many K blocks in the split tiles
 *                 as clusters in the grid, else the launch runs unsplit.
 *   workspace / workspace_bytes  device memory for stream_k (NULL: no
 *                 split): at least gemm_streamk_workspace_size() bytes,
 *                 256-byte aligned, set to zero once before its first use
 *                 (the library leaves it reusable: each launch tags its
 *                 flags with a new value). Calls that may run at the same
 *                 time, on different streams, need different workspaces.
 *   mma_ws        weight-stationary MMA (tcgen05.mma.ws, "How cta_group Sets
 *                 the Operation Scope": one of the choices that fix the
 *                 accumulator layout): 0 the library chooses, 1 use it,
 *                 -1 do not. It serves tiles of 32 or 64 rows of single
 *                 problems with 16-bit operands on one CTA (tile_n 128 or 256
 *                 for 64 rows, 256 for 32); its accumulator is spread over
 *                 the four TMEM lane quarters by column parts, so all four
 *                 epilogue warps store full 32-row chunks. Other tiles with
 *                 mma_ws 1 return GEMM_ERR_UNSUPPORTED.
 *   multicast_b   single-CTA (cta_group::1) tiles 256 wide (128 or 256 rows),
 *                 or 224 wide with 256 rows and K-major B,
 *                 run in clusters of two CTAs on vertically adjacent tiles
 *                 that share their B panel: each CTA loads half of every B
 *                 stage and TMA multicasts it into both CTAs' shared memory,
 *                 so each CTA reads half as many B bytes from L2; each CTA's
 *                 MMA completion releases the stage in both. 0 the library
 *                 chooses (256 x 256 tiles of more than 256 rows in all; 128-row
 *                 tiles when B is MN-major or A and B overflow L2), 1 use it,
 *                 -1 do not; other tiles with 1 return GEMM_ERR_UNSUPPORTED.
 *                 Multicast stays within this GPU's memory (the operands of
 *                 one call).
 */
typedef struct {
    int cta_group;
    int tile_m;
    int tile_n;
    int block_k;
    int swizzle_a;
    int swizzle_b;
    int epilogue_swizzle;
    int max_ctas;
    int group_m;
    int timeout_ms;
    int flags;
    unsigned long long *stats;
    int stream_k;
    void *workspace;
    size_t workspace_bytes;
    int mma_ws;
    int multicast_b;
} gemm_options_t;

/* Bytes of stream-K workspace for any single GEMM on the current device:
 * one 4 x uint32 flag row and one 256 x 256 fp32 partial-sum slot per SM
 * (the largest tile; 128-row tiles use half of each slot).
 * 0 if the device cannot be queried. */
size_t gemm_streamk_workspace_size(void);

/* One problem of a grouped call. All share the call's majors, types,
 * alpha and beta; each has its own sizes, pointers and leading dims. */
typedef struct {
    int64_t M, N, K;
    const void *A;
    const void *B;
    const void *C;
    void *D;
    int64_t lda, ldb, ldc, ldd;
} gemm_problem_t;

/*
 * gemm_bf16 / gemm_f16: one GEMM, inputs bf16 / fp16, fp32 accumulation,
 * output d_type. Tiles of 128 x tile_n (256 x tile_n for CTA pairs) are
 * dealt round-robin to a persistent grid of one CTA per SM; operands reach
 * shared memory by TMA in swizzled layouts, tcgen05.mma accumulates in
 * Tensor Memory, and a warp-specialised epilogue applies alpha/beta and
 * stores D by TMA.
 */
gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K,
                        const void *A, gemm_major_t a_major, int64_t lda,
                        const void *B, gemm_major_t b_major, int64_t ldb,
                        const void *C, int64_t ldc,
                        void *D, int64_t ldd, gemm_out_t d_type,
                        float alpha, float beta, gemm_stream_t stream);

gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K,
                       const void *A, gemm_major_t a_major, int64_t lda,
                       const void *B, gemm_major_t b_major, int64_t ldb,
                       const void *C, int64_t ldc,
                       void *D, int64_t ldd, gemm_out_t d_type,
                       float alpha, float beta, gemm_stream_t stream);

/* The same with explicit options (opts may be NULL). in_type: 0 fp16, 1 bf16,
 * 2 TF32: A and B hold fp32 words (leading dimensions in elements, multiples
 * of 4) and tcgen05 kind::tf32 multiplies their TF32 part -- sign, exponent
 * and the top 10 fraction bits; the low 13 fraction bits are dropped (a
 * reading of the hardware, pinned by the tests). MN-major TF32 operands are
 * staged in the 128-byte swizzle with 32-byte atoms (GEMM_SWIZZLE_128B_ATOM32,
 * descriptor code 1): kind::tf32 reads an MN-major operand in that layout and
 * as zeros in SW128 (measured); K-major TF32 operands use the 32/64/128-byte
 * swizzles of the 16-bit types. */
gemm_status_t gemm_ex(int in_type, int64_t M, int64_t N, int64_t K,
                      const void *A, gemm_major_t a_major, int64_t lda,
                      const void *B, gemm_major_t b_major, int64_t ldb,
                      const void *C, int64_t ldc,
                      void *D, int64_t ldd, gemm_out_t d_type,
                      float alpha, float beta, const gemm_options_t *opts,
                      gemm_stream_t stream);

/* 8-bit float operand formats (tcgen05.mma kind::f8f6f4). */
typedef enum { GEMM_FP8_E4M3 = 0, GEMM_FP8_E5M2 = 1 } gemm_fp8_t;

/*
 * gemm_fp8 / gemm_fp8_ex: the same GEMM with 8-bit float operands, A and B
 * each E4M3 or E5M2 (they may differ), fp32 accumulation, output d_type.
 * The descriptors are the same as for 16-bit operands: one 16-byte core-matrix
 * cell holds 16 fp8 values ("LBO, SBO and SWZ for a tcgen05 tile", section 4)
 * and one MMA consumes 32 of them along K. Leading dimensions lda and ldb are
 * counted in elements (bytes) and must be multiples of 16; the other rules
 * are those above. opts may be NULL.
 */
gemm_status_t gemm_fp8(int64_t M, int64_t N, int64_t K,
                       const void *A, gemm_fp8_t a_format, gemm_major_t a_major, int64_t lda,
                       const void *B, gemm_fp8_t b_format, gemm_major_t b_major, int64_t ldb,
                       const void *C, int64_t ldc,
                       void *D, int64_t ldd, gemm_out_t d_type,
                       float alpha, float beta, gemm_stream_t stream);

gemm_status_t gemm_fp8_ex(int64_t M, int64_t N, int64_t K,
                          const void *A, gemm_fp8_t a_format, gemm_major_t a_major, int64_t lda,
                          const void *B, gemm_fp8_t b_format, gemm_major_t b_major, int64_t ldb,
                          const void *C, int64_t ldc,
                          void *D, int64_t ldd, gemm_out_t d_type,
                          float alpha, float beta, const gemm_options_t *opts,
                          gemm_stream_t stream);

/*
 * gemm_mxfp8: block-scaled fp8 GEMM (MXFP8: tcgen05 kind::mxf8f6f4 with
 * scale_vec::1X; "06 Blackwell Tensor Core - tcgen05 MMA", block-scaled
 * MMA: scale factors go from global memory to shared memory, then by
 * tcgen05.cp into TMEM, where the MMA reads them next to A and B).
 *   D = alpha * sum_k (sa[m, k/32] * A[m,k]) * (sb[n, k/32] * B[k,n]) + beta * C
 * A and B are E4M3 or E5M2 exactly as for gemm_fp8_ex; every 32 consecutive
 * elements of K of a row of A (column of B) share one scale, an 8-bit E8M0
 * code e meaning 2^(e - 127) (255 is NaN). The scales are stored in 512-byte
 * atoms, each covering 128 rows (of A; columns of B) x 4 scale blocks (128
 * elements of K): row r and K element k live in atom
 * (r / 128) * ceil(K / 128) + k / 128, at byte
 * 16 * (r % 32) + 4 * ((r % 128) / 32) + (k / 32) % 4 of it -- the layout
 * tcgen05.cp copies into TMEM, replicated over the four lane quarters.
 * SFA and SFB are device pointers, 16-byte aligned, of
 * gemm_mx_scale_bytes(M, K) and gemm_mx_scale_bytes(N, K) bytes; entries
 * for rows past M (N) or blocks past K are read and multiply only zeros, so
 * they must not be NaN (255).
 * Tiles: CTA pairs sharing a 256 x 256 tile (the default from M, N >= 2048;
 * one accumulator buffer, so each tile's epilogue is not overlapped and
 * stream_k is not applied), single CTAs of 128 x 128 (the default below
 * that), or pairs sharing 256 x 128 (cta_group 2 with tile_n 128). In a
 * pair each CTA holds the scales of its own A rows and a copy of all the
 * tile's B scales. 256
 * elements of K per pipeline stage (single CTAs may ask block_k = 128);
 * options asking for other tiles return GEMM_ERR_UNSUPPORTED. stream_k
 * applies as for gemm_ex.
 */
gemm_status_t gemm_mxfp8(int64_t M, int64_t N, int64_t K,
                         const void *A, gemm_fp8_t a_format, gemm_major_t a_major, int64_t lda,
                         const void *SFA,
                         const void *B, gemm_fp8_t b_format, gemm_major_t b_major, int64_t ldb,
                         const void *SFB,
                         const void *C, int64_t ldc,
                         void *D, int64_t ldd, gemm_out_t d_type,
                         float alpha, float beta, const gemm_options_t *opts,
                         gemm_stream_t stream);

/* Bytes of one scale tensor of gemm_mxfp8 for `rows` rows (M for SFA, N for
 * SFB) and K: ceil(rows / 128) * ceil(K / 128) * 512; 0 if either is <= 0. */
size_t gemm_mx_scale_bytes(int64_t rows, int64_t K);

/* Block-scaled fp4 formats of gemm_fp4 (E2M1 elements in both). */
typedef enum {
    GEMM_FP4_NVFP4 = 0, /* one UE4M3 scale per 16 elements of K (kind::mxf4nvf4, scale_vec::4X) */
    GEMM_FP4_MXFP4 = 1  /* one E8M0 scale per 32 elements of K (kind::mxf4, scale_vec::2X) */
} gemm_fp4_scale_t;

/*
 * gemm_fp4: block-scaled fp4 GEMM, the fp4 members of the block-scaled MMA
 * family of "06 Blackwell Tensor Core - tcgen05 MMA" (scales through
 * tcgen05.cp into TMEM, as for gemm_mxfp8).
 *   D = alpha * sum_k (sa[m, k/b] * A[m,k]) * (sb[n, k/b] * B[k,n]) + beta * C
 * with block b = 16 (NVFP4) or 32 (MXFP4). A (M x K) and B (stored N x K)
 * are K-major, E2M1 packed two to a byte: element 2i of a row in the low
 * nibble of byte i, 2i+1 in the high nibble. K, lda and ldb count elements;
 * K must be even and lda, ldb multiples of 32 (16-byte rows). Scale codes:
 * UE4M3 (unsigned E4M3: 2^(e-7) * (1 + m/8), e = 0 subnormal) for NVFP4,
 * E8M0 (2^(e-127)) for MXFP4, in the 512-byte atoms of gemm_mxfp8, one atom
 * per 128 rows x 4 blocks: row r and element k live in atom
 * (r / 128) * ceil(K / (4b)) + k / (4b), at byte
 * 16 * (r % 32) + 4 * ((r % 128) / 32) + (k / b) % 4. SFA and SFB hold
 * gemm_fp4_scale_bytes(M, K, kind) and gemm_fp4_scale_bytes(N, K, kind)
 * bytes, 16-byte aligned; entries for rows past M (N) or blocks past K
 * multiply only zeros but must be finite scales (a NaN code there, UE4M3
 * 0x7F or E8M0 255, makes the whole result NaN). Tiles: 256 x 256 CTA pairs
 * with one accumulator buffer (default from M, N >= 2048; cta_group 2) or
 * single CTAs of 128 x 128; stream_k (single CTAs)
 * applies as for gemm_ex; other tile options return GEMM_ERR_UNSUPPORTED.
 */
gemm_status_t gemm_fp4(int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda, const void *SFA,
                       const void *B, int64_t ldb, const void *SFB,
                       gemm_fp4_scale_t kind,
                       const void *C, int64_t ldc,
                       void *D, int64_t ldd, gemm_out_t d_type,
                       float alpha, float beta, const gemm_options_t *opts,
                       gemm_stream_t stream);

/* Bytes of one scale tensor of gemm_fp4 for `rows` rows and K elements:
 * ceil(rows / 128) * ceil(K / (4 * block)) * 512; 0 for bad arguments. */
size_t gemm_fp4_scale_bytes(int64_t rows, int64_t K, gemm_fp4_scale_t kind);

/*
 * Grouped GEMM: num_problems independent problems in one launch. The
 * host list is read during the call; the library writes the device-side
 * problem list, one TMA descriptor per operand per problem and the tile
 * prefix sums into `workspace` (device memory owned by the caller, at
 * least gemm_grouped_workspace_size(num_problems) bytes, 128-byte
 * aligned) with an asynchronous copy on `stream`, then launches one
 * persistent kernel whose scheduler walks the concatenated tile list.
 * The workspace must stay untouched until the launch completes.
 */
size_t gemm_grouped_workspace_size(int num_problems);

gemm_status_t gemm_bf16_grouped(const gemm_problem_t *problems, int num_problems,
                                gemm_major_t a_major, gemm_major_t b_major,
                                gemm_out_t d_type, float alpha, float beta,
                                void *workspace, size_t workspace_bytes,
                                gemm_stream_t stream);

gemm_status_t gemm_f16_grouped(const gemm_problem_t *problems, int num_problems,
                               gemm_major_t a_major, gemm_major_t b_major,
                               gemm_out_t d_type, float alpha, float beta,
                               void *workspace, size_t workspace_bytes,
                               gemm_stream_t stream);

/* The grouped call with explicit options (opts may be NULL; tile_m, timeout
 * and flags as for gemm_ex). in_type: 0 fp16, 1 bf16. Without a cta_group
 * option, lists whose widest problem has N >= 2048 and whose tallest has
 * M >= 256 run on CTA pairs (256 x 256 tiles), others on single CTAs. */
gemm_status_t gemm_grouped_ex(int in_type, const gemm_problem_t *problems, int num_problems,
                              gemm_major_t a_major, gemm_major_t b_major,
                              gemm_out_t d_type, float alpha, float beta,
                              void *workspace, size_t workspace_bytes,
                              const gemm_options_t *opts, gemm_stream_t stream);

/*
 * gemm_bf16_grouped_noalloc: the grouped bf16 GEMM for callers that cannot
 * allocate device memory when they launch it: programs whose allocator has
 * reserved the whole device and forbids side allocations, plug-ins that a
 * host runtime hands only their input and output buffers, and real-time
 * loops that may not block in the driver's allocator (cudaMalloc can
 * synchronise the device). There is no counterpart on the pages; it is a
 * service of this library. Instead of a caller workspace, the problem table
 * and TMA descriptors go into a fixed array inside the library (about 68 KB,
 * room for GEMM_NOALLOC_MAX_PROBLEMS problems) that every GPU which loads the
 * library keeps until the process exits. The call allocates no device
 * memory and calls no allocating library routine; the table is staged in a
 * fixed host array and copied to the device array with cudaMemcpyAsync on
 * `stream` before the kernel launch.
 *   - Same arguments and results as gemm_bf16_grouped, minus the workspace.
 *   - num_problems > GEMM_NOALLOC_MAX_PROBLEMS returns GEMM_ERR_INVALID_ARG
 *     and enqueues nothing.
 *   - Set-up: the first call on a device looks up the array's device address
 *     there (cudaGetSymbolAddress, with that device current) and keeps it.
 *     Make that first call before any stream capture begins.
 *   - All calls share the array and each call rewrites the part it uses, so
 *     calls whose kernels may overlap on the GPU (other streams, or no
 *     ordering between them) race: order them on one stream or synchronise.
 */
#define GEMM_NOALLOC_MAX_PROBLEMS 128

gemm_status_t gemm_bf16_grouped_noalloc(const gemm_problem_t *problems, int num_problems,
                                        gemm_major_t a_major, gemm_major_t b_major,
                                        gemm_out_t d_type, float alpha, float beta,
                                        gemm_stream_t stream);

/* Synchronises `stream`, reads the device status word of this library,
 * clears it, and returns GEMM_OK or GEMM_ERR_TIMEOUT (GEMM_ERR_CUDA if the
 * read fails). `detail` (may be NULL) receives the raw word: bits 0-7 the
 * role that gave up (1 producer, 2 MMA, 3 epilogue, 4 scale copier of the
 * block-scaled kinds, 5 launch setup: 10 in bits 8-15 means the dynamic
 * shared memory was not 1024-byte aligned), bits 8-15 the wait. */
gemm_status_t gemm_last_device_status(gemm_stream_t stream, uint32_t *detail);

const char *gemm_status_string(gemm_status_t status);

/* Number of this library's kernels launched since the library loaded. */
uint64_t gemm_launch_count(void);

/* ---------------------------------------------------------------------
 * Inspection entry points (tests): they expose the device-side builders
 * so their output can be compared bit for bit with an independent model.
 * ------------------------------------------------------------------- */

/*
 * Runs the device-side descriptor builder on the GPU and writes, for each
 * of the n_slices K=16 slices of one operand stage, the 64-bit shared-
 * memory matrix descriptor the GEMM kernel would hand to tcgen05.mma
 * ("LBO, SBO and SWZ for a tcgen05 tile", section 3: start, LBO, SBO, MBO
 * and SWZ fields), followed by the 32-bit instruction descriptor for
 * (M = 128 * cta_group, N = tile_n, in_type, f32 accumulate, majors) in the
 * low half of word n_slices. `out` is device memory of n_slices + 1 words.
 *   major: gemm_major_t of the operand; swizzle: gemm_swizzle_t (not AUTO);
 *   rows: MN extent of the stage (128 for A; tile_n or tile_n/2 for B);
 *   bk: K extent of the stage (32 or 64); stage_addr: shared-memory byte
 *   address of the stage (1024-aligned).
 */
gemm_status_t gemm_debug_descriptors(int major, int swizzle, int rows, int bk,
                                     uint32_t stage_addr, int n_slices,
                                     int cta_group, int tile_n, int in_type,
                                     int a_major, int b_major,
                                     uint64_t *out, gemm_stream_t stream);

/*
 * Loads one operand stage exactly as the GEMM producer does (TMA boxes in
 * the given swizzle into a 1024-aligned shared buffer) and copies the raw
 * shared-memory bytes to `out` (device memory, rows * bk * 2 bytes).
 *   src: device matrix of 16-bit elements, stored with leading dimension ld
 *   (K-major: rows_total x K with K contiguous; MN-major: K x rows_total
 *   with the MN index contiguous); (mn0, k0): the stage's origin.
 */
gemm_status_t gemm_debug_stage_image(const void *src, int major, int swizzle,
                                     int64_t rows_total, int64_t k_total, int64_t ld,
                                     int rows, int bk, int64_t mn0, int64_t k0,
                                     void *out, gemm_stream_t stream);

/*
 * Host-side tile plan (no GPU needed): the configuration a call would launch
 * on a device with `sms` SMs. kind: 0 fp16/bf16, 1 fp8, 2 MXFP8, 3 NVFP4,
 * 4 MXFP4 (K in elements), 5 TF32; grouped: nonzero for the grouped entry
 * points.
 * Writes 10 int32: cta_group, tile N, K per stage (bytes for fp4), rows per
 * CTA, swizzle bits of A and B (0 none, 1 32B, 2 64B, 3 128B, 4 128B with
 * 32-byte atoms), epilogue swizzle, group height, 1 when the tiles use
 * tcgen05.mma.ws, and 1 when two CTAs share B by multicast. Returns the
 * status the call's planning would.
 */
gemm_status_t gemm_debug_plan(int64_t M, int64_t N, int64_t K, int kind, int a_major, int b_major, int grouped,
                              const gemm_options_t *opts, int sms, int32_t *out);

/*
 * Host-side listing of the stream-K schedule (no GPU needed): the split the
 * library would choose for `tiles` tiles of `kb_per_tile` K blocks on a
 * grid of `clusters` clusters under stream_k `mode`, and the units of
 * cluster `cluster` in the order its roles run them -- the same code the
 * kernel's roles execute. Writes 6 int32 per unit to `out` (room for
 * max_units): tile, first K block, end K block (-1: the whole tile), kind
 * (0 whole, 1 contributor, 2 head), and for a head the first and last
 * contributing cluster (else 0, -1). Returns the number of units, or -1
 * when the launch would stay data-parallel (no units listed).
 */
int gemm_debug_streamk_units(int mode, int64_t tiles, int clusters, int kb_per_tile, int cluster,
                             int32_t *out, int max_units);

/* Test hook: the next GEMM launch makes its MMA warp wait on a barrier
 * that nothing arrives at, with a wait bound of `timeout_ms`; every role
 * then gives up and the kernel exits with GEMM_ERR_TIMEOUT recorded. */
void gemm_debug_inject_timeout(int timeout_ms);

/* The same for a chosen role: 1 the TMA producer (in both CTAs of a pair,
 * before it issues any load), 2 the MMA issuer. Other roles are ignored. The
 * status word then names that role with wait code 6 (injected). */
void gemm_debug_inject_timeout_at(int timeout_ms, int role);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
