/*
 * tkg_gemm.h -- C ABI of libtkg.so: dense and block-scaled GEMM on one GB300
 * (sm_103a), plus the quantisers and the scale-layout conversion that feed it.
 *
 *   D = alpha_eff * A * B^T
 *
 * A is M x K and B is N x K, both row-major ("K-major", K contiguous); D is
 * M x N row-major BF16.  Products are accumulated in FP32 on the tensor cores;
 * D is alpha_eff * acc rounded to nearest-even BF16.  The three operand formats
 * are the BF16 / MXFP8 / NVFP4 GEMMs of "ThunderKittens 2.0 GPU Kernel优化"
 * (yunpan.plus write-up of the HazyResearch TK 2.0 release, opening section and
 * its table of updates); the pages name the formats, these declarations fix
 * their layouts.
 *
 * Conventions for every entry point below:
 *  - Pointers named A, B, D, X, Q, sfa, sfb, sf, src, dst are DEVICE pointers
 *    owned by the caller; the library keeps no reference after the call.
 *  - Calls are asynchronous on `stream` and return after enqueueing work.
 *    Device-side failures (a bounded wait that ran out) are reported by
 *    tkg_get_device_status().
 *  - Stream order holds as for any kernel: a GEMM reads what earlier work on
 *    the stream wrote, and later work sees its D.  GEMM launches carry the
 *    programmatic-dependent-launch attribute, so a GEMM's set-up (and L2
 *    prefetches of its first operand tiles) may start while the previous
 *    kernel finishes; every read of operands, scales and tensor scales, and
 *    every store of D, waits for that kernel to complete.
 *  - Arguments are checked before anything is launched: negative sizes or a
 *    null pointer give TKG_ERR_INVALID_ARG, a base address or row pitch that
 *    is not a multiple of 16 bytes gives TKG_ERR_ALIGNMENT, shapes the kernels
 *    do not handle give TKG_ERR_UNSUPPORTED.  A CUDA error while enqueueing
 *    gives TKG_ERR_CUDA.  There is no CPU fallback.
 *  - m == 0 or n == 0 is an empty GEMM (nothing is written); k == 0 writes
 *    zeros to D (an empty sum).
 *
 * Block-scaled scale factors use the TILED layout (tkg_scale_bytes): for a
 * matrix with R rows and KB = ceil(K / bs) scale blocks per row (bs = 32 for
 * MXFP8, 16 for NVFP4), scale (r, kb) is the byte at
 *
 *     ((r / 128) * KA + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4
 *
 * with KA = ceil(KB / 4).  Each 512-byte atom holds 128 rows x 4 blocks in the
 * order the tensor cores read scales from tensor memory, so the kernel moves
 * atoms from HBM to shared memory to tensor memory without rearranging bytes.
 * Rows beyond R and blocks beyond KB are padding: padding blocks inside a row
 * must hold a finite scale code (zero is recommended; the quantisers and
 * tkg_scales_to_tiled write zeros).  tkg_scales_to_tiled() converts a
 * row-major scale matrix into this layout.
 */
#ifndef TKG_GEMM_H
#define TKG_GEMM_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TKG_OK = 0,
  TKG_ERR_INVALID_ARG = 1,
  TKG_ERR_ALIGNMENT = 2,
  TKG_ERR_UNSUPPORTED = 3,
  TKG_ERR_CUDA = 4,
  TKG_ERR_TIMEOUT = 5,
  TKG_ERR_CHECK = 6   /* an internal invariant failed in a check build (libtkg_check.so) */
} tkg_status;

/* BF16 GEMM ("ThunderKittens 2.0", opening section: BF16 GEMM on B200).
 * A: m x k bfloat16, B: n x k bfloat16, D: m x n bfloat16, all row-major.
 * Requires k % 8 == 0 and n % 8 == 0 (16-byte row pitches) and 16-byte
 * aligned A, B, D.  D = bf16_rn(alpha * sum_k A[i][k] * B[j][k]). */
tkg_status tkg_gemm_bf16(int m, int n, int k, const void *A, const void *B, void *D, float alpha,
                         cudaStream_t stream);

/* MXFP8 GEMM ("ThunderKittens 2.0", table of updates: MXFP8 support).
 * A: m x k bytes (FP8 E4M3), B: n x k bytes (E4M3), sfa / sfb: E8M0 scale
 * codes (2^(c-127)), one per 1 x 32 block along K, tiled layout (bs = 32),
 * tkg_scale_bytes(m, k, 32) / tkg_scale_bytes(n, k, 32) bytes.
 * Requires k % 32 == 0, n % 8 == 0, 16-byte aligned pointers.
 * D[i][j] = bf16_rn(alpha * sum_k a_ik * sa(i, k/32) * b_jk * sb(j, k/32)). */
tkg_status tkg_gemm_mxfp8(int m, int n, int k, const void *A, const void *B, const void *sfa, const void *sfb,
                          void *D, float alpha, cudaStream_t stream);

/* NVFP4 GEMM ("ThunderKittens 2.0", table of updates: NVFP4 support; §二 2.1
 * on its scale path).  A: m x k/2 bytes, B: n x k/2 bytes, two FP4 E2M1 codes
 * per byte, element 2j in the low nibble of byte j.  sfa / sfb: UE4M3 scale
 * codes, one per 1 x 16 block along K, tiled layout (bs = 16).
 * tensor_scale_a / tensor_scale_b: device pointers to the FP32 per-tensor
 * scales (either may be NULL, meaning 1.0).  The kernel forms
 * alpha_eff = fp32(fp32(alpha * tA) * tB).  Requires k % 32 == 0, n % 8 == 0.
 * D[i][j] = bf16_rn(alpha_eff * sum_k a_ik * sa(i, k/16) * b_jk * sb(j, k/16)). */
tkg_status tkg_gemm_nvfp4(int m, int n, int k, const void *A, const void *B, const void *sfa, const void *sfb,
                          const float *tensor_scale_a, const float *tensor_scale_b, void *D, float alpha,
                          cudaStream_t stream);

/* The three GEMMs above on matrices with row pitches (views into larger
 * buffers, or rows padded for alignment).  Same products, scales and checks,
 * except that row i of A starts lda units after row i-1 and row j of B ldb
 * units after row j-1, where a unit is an element of the operand's storage
 * (a bfloat16 for BF16; a byte, i.e. one E4M3 code or two E2M1 codes, for
 * MXFP8 and NVFP4), and row i of D starts ldd bfloat16 elements after row i-1.
 * Requires lda, ldb >= the row length (k, or k/2 bytes for NVFP4) and ldd >= n
 * (else TKG_ERR_INVALID_ARG), and pitches that are multiples of 16 bytes (else
 * TKG_ERR_ALIGNMENT); bytes between rows are neither read (A, B) nor written
 * (D).  k == 0 writes zeros to the m x n block of D.
 * Pitches that are an odd multiple of 16 bytes start every other row 16 bytes
 * off a 32-byte boundary, so its 128-byte pieces span five 32-byte sectors
 * instead of four: such GEMMs run 20-27% slower than with 32-byte multiples. */
tkg_status tkg_gemm_bf16_strided(int m, int n, int k, const void *A, int lda, const void *B, int ldb, void *D, int ldd,
                                 float alpha, cudaStream_t stream);
tkg_status tkg_gemm_mxfp8_strided(int m, int n, int k, const void *A, int lda, const void *B, int ldb, const void *sfa,
                                  const void *sfb, void *D, int ldd, float alpha, cudaStream_t stream);
tkg_status tkg_gemm_nvfp4_strided(int m, int n, int k, const void *A, int lda, const void *B, int ldb, const void *sfa,
                                  const void *sfb, const float *tensor_scale_a, const float *tensor_scale_b, void *D,
                                  int ldd, float alpha, cudaStream_t stream);

/* Grouped GEMM, the mixture-of-experts form named as work in progress in
 * "ThunderKittens 2.0 GPU Kernel优化" (section after Figure 1: grouped GEMM
 * kernels under development).  The pages give no interface; this one keeps the
 * plain GEMM's layouts per group.
 *
 * groups (1..128) groups of rows; m_sizes: HOST array of the groups' row
 * counts (each >= 0, read during the call).  Group g owns the M_g = m_sizes[g]
 * consecutive rows of A and D starting at row o_g = m_sizes[0] + ... +
 * m_sizes[g-1], and multiplies them by its own n x k matrix B_g:
 *   D[o_g + i][j] = bf16_rn(alpha_g * sum_k A[o_g + i][k] * B_g[j][k]).
 * A: (sum M_g) x k, D: (sum M_g) x n, B: groups x n x k (B_g at row g * n),
 * element types and per-format requirements as in the plain GEMMs; rows of D
 * outside the groups' ranges are not written.
 * Block scales: SFA holds each group's scales as its own tiled buffer of
 * tkg_scale_bytes(M_g, k, bs) bytes, one after another (group g at the sum of
 * the earlier groups' sizes; tkg_grouped_scale_bytes gives the total); SFB
 * holds groups tiled buffers of tkg_scale_bytes(n, k, bs) bytes each.
 * NVFP4: tensor_scale_a is NULL or one FP32 for all of A, tensor_scales_b NULL
 * or one FP32 per group; alpha_g = fp32(fp32(alpha * tA) * tB[g]).
 * Errors: groups < 1, m_sizes NULL or a negative size -> TKG_ERR_INVALID_ARG;
 * groups > 128 -> TKG_ERR_UNSUPPORTED; otherwise as the plain GEMMs.  All
 * groups empty or n == 0: nothing to do, TKG_OK. */
tkg_status tkg_gemm_grouped_bf16(int groups, const int *m_sizes, int n, int k, const void *A, const void *B, void *D,
                                 float alpha, cudaStream_t stream);
tkg_status tkg_gemm_grouped_mxfp8(int groups, const int *m_sizes, int n, int k, const void *A, const void *B,
                                  const void *sfa, const void *sfb, void *D, float alpha, cudaStream_t stream);
tkg_status tkg_gemm_grouped_nvfp4(int groups, const int *m_sizes, int n, int k, const void *A, const void *B,
                                  const void *sfa, const void *sfb, const float *tensor_scale_a,
                                  const float *tensor_scales_b, void *D, float alpha, cudaStream_t stream);

/* Bytes of a grouped SFA buffer: the sum over groups of
 * tkg_scale_bytes(m_sizes[g], k, block).  0 for invalid arguments. */
size_t tkg_grouped_scale_bytes(int groups, const int *m_sizes, int k, int block);

/* Grouped GEMM with the group sizes in DEVICE memory (for instance written by
 * a router kernel earlier on the stream; read after the work already queued
 * on `stream`, so no host synchronisation is needed).  Same product and
 * layouts as tkg_gemm_grouped_*, except:
 *  - m_sizes_dev: device array of `groups` int32 row counts (4-byte aligned);
 *    a negative count is taken as 0.
 *  - m_capacity: rows allocated for A and D (and the bound the sizes are
 *    expected to respect); rows of A past it are never read and rows of D past
 *    it never written, whatever the sizes say.
 *  - SFA: per-group tiled buffers back to back as before; the buffer must hold
 *    tkg_grouped_dev_scale_bytes(groups, m_capacity, k, bs) bytes (the most any
 *    split of m_capacity rows into `groups` groups needs).
 *  - k == 0 gives TKG_ERR_UNSUPPORTED (which rows to zero is known only on the
 *    device).  m_capacity == 0 or n == 0: nothing to do.
 *  - Runs the static persistent schedule (the tile count is found on the
 *    device). */
tkg_status tkg_gemm_grouped_dev_bf16(int groups, const int *m_sizes_dev, int m_capacity, int n, int k,
                                     const void *A, const void *B, void *D, float alpha, cudaStream_t stream);
tkg_status tkg_gemm_grouped_dev_mxfp8(int groups, const int *m_sizes_dev, int m_capacity, int n, int k,
                                      const void *A, const void *B, const void *sfa, const void *sfb, void *D,
                                      float alpha, cudaStream_t stream);
tkg_status tkg_gemm_grouped_dev_nvfp4(int groups, const int *m_sizes_dev, int m_capacity, int n, int k,
                                      const void *A, const void *B, const void *sfa, const void *sfb,
                                      const float *tensor_scale_a, const float *tensor_scales_b, void *D,
                                      float alpha, cudaStream_t stream);

/* Bytes an SFA buffer needs for tkg_gemm_grouped_dev_* with up to m_capacity
 * rows in `groups` groups: tkg_scale_bytes(m_capacity, k, block) plus
 * groups * tkg_scale_bytes(128, k, block).  0 for invalid arguments. */
size_t tkg_grouped_dev_scale_bytes(int groups, int m_capacity, int k, int block);

/* A list of independent GEMMs run by one persistent launch ("ThunderKittens
 * 2.0 GPU Kernel优化", table of updates: cluster-launch-control scheduling and
 * programmatic dependent launch, named there as the means for back-to-back
 * small GEMMs).  Each entry is a whole GEMM of its own, with the plain
 * entry point's product, layouts and requirements for its format:
 *   D_e = bf16_rn(alpha_e' * A_e * B_e^T),  A_e: m x k, B_e: n x k, D_e: m x n,
 * alpha_e' = alpha (BF16, MXFP8) or fp32(fp32(alpha * tA) * tB) (NVFP4, either
 * pointer may be NULL meaning 1.0).  All entries' output tiles form one tile
 * list, so small GEMMs -- the projections of one decode step, a batch of
 * 512^3 products -- fill the SMs together and pay one launch's fixed cost.
 *  - gemms: HOST array of `count` descriptors (1..16), read during the call.
 *    Entries with m == 0 or n == 0 are skipped; k == 0 writes zeros to D.
 *  - sfa / sfb: tiled scales as in tkg_gemm_mxfp8 / tkg_gemm_nvfp4 (ignored
 *    for BF16); tensor_scale_a / tensor_scale_b: NVFP4 only.
 *  - The outputs must not overlap one another or any entry's inputs.
 * Errors: count outside 1..16 or gemms NULL -> TKG_ERR_INVALID_ARG
 * (count > 16: TKG_ERR_UNSUPPORTED); an entry failing the plain entry point's
 * checks -> that entry point's error, and nothing is launched. */
typedef struct {
  int m, n, k;
  const void *A, *B;
  const void *sfa, *sfb;
  const float *tensor_scale_a, *tensor_scale_b;
  void *D;
  float alpha;
} tkg_gemm_desc;

tkg_status tkg_gemm_list_bf16(int count, const tkg_gemm_desc *gemms, cudaStream_t stream);
tkg_status tkg_gemm_list_mxfp8(int count, const tkg_gemm_desc *gemms, cudaStream_t stream);
tkg_status tkg_gemm_list_nvfp4(int count, const tkg_gemm_desc *gemms, cudaStream_t stream);

/* BF16 GEMM on operands in HOST memory (the same product as tkg_gemm_bf16;
 * no counterpart on the pages, which time device-resident GEMMs only).
 * A_host (m x k), B_host (n x k): bfloat16, row-major, read; D_host (m x n):
 * written.  A_dev, B_dev, D_dev: caller-owned device buffers of the same
 * sizes used as staging (16-byte aligned); their contents afterwards are
 * unspecified except D_dev = D.  The call copies A and B in bands of rows,
 * alternating, on one internal stream; each band unlocks a rectangle of D (the
 * new band against the other operand's bands already copied), whose GEMM runs
 * on `stream` once the band has landed and which goes back on a second
 * internal stream as soon as that GEMM is done, so the copies overlap the
 * GEMM; host buffers must be page-locked (cudaHostAlloc / cudaHostRegister)
 * for that overlap.  Asynchronous: everything starts after
 * the work already queued on `stream`, and work queued on `stream` afterwards
 * starts after D_host is written.  Concurrent calls from several threads are
 * serialised while they enqueue.  Checks and errors as tkg_gemm_bf16. */
tkg_status tkg_gemm_bf16_from_host(int m, int n, int k, const void *A_host, const void *B_host, void *D_host,
                                   void *A_dev, void *B_dev, void *D_dev, float alpha, cudaStream_t stream);

/* BF16 GEMM that allocates nothing, for callers that cannot call cudaMalloc:
 * runtimes that reserve all of their device memory at start-up and forbid
 * allocation afterwards, or that run under a memory budget where an
 * allocation hidden inside a library call must not happen.  (No counterpart
 * on the pages: this is a property of the library, not of the method.)
 *
 * Same arguments, layouts, checks and result as tkg_gemm_bf16, and the same
 * CTA-pair kernel on its static persistent schedule.  Its scratch -- the
 * status word the kernel sets when a bounded wait runs out -- lives in a fixed
 * 256-byte array that is part of the library image (each GPU that loads the
 * library keeps it until the process exits) instead of memory obtained with
 * cudaMalloc.  The kernel needs 4 bytes of it whatever m, n and k are; a call
 * whose scratch need exceeded the array would return TKG_ERR_UNSUPPORTED.
 *  - The first call on a device does one-time set-up there (it looks up the
 *    array's device address, clears the array on `stream` and sets the
 *    kernel's shared-memory limit); make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one array, so calls that overlap on the
 *    GPU race on it: order them on one stream or with events.
 *  - A timed-out wait sets the array's status word, which no call clears on
 *    entry; tkg_get_device_status reads it and clears it (allocating nothing),
 *    as it does the library's own word.  D is then unspecified.
 *  - Options set with tkg_set_option apply as to tkg_gemm_bf16, except that the
 *    schedule is always the static one. */
tkg_status tkg_gemm_bf16_noalloc(int m, int n, int k, const void *A, const void *B, void *D, float alpha,
                                 cudaStream_t stream);

/* Check builds.  `python -m dense_block_scaled_gb300.build --check` builds the
 * same library as libtkg_check.so with every kernel verifying its internal
 * invariants (tensor-memory column ranges of each MMA, scale copy and
 * accumulator load; ring-slot, accumulator, tile, group and GEMM-list
 * indices; the 16-byte alignment of TMA x coordinates).  A failed invariant
 * skips the access it guards and is reported by tkg_get_device_status as
 * TKG_ERR_CHECK; nothing traps.  Meant for testing, not for speed.
 *
 * Synchronises `stream`, then reads and clears the current device's status
 * words: the library's own (created by the first allocating entry point on the
 * device) and that of tkg_gemm_bf16_noalloc (once set up on the device).
 * Returns TKG_ERR_TIMEOUT if a kernel's bounded wait ran out since the last
 * call (its output is then unspecified), TKG_ERR_CHECK if an invariant failed
 * (check builds), TKG_ERR_CUDA on a CUDA error, TKG_OK otherwise.  Allocates nothing: a word that does not exist yet reads as
 * clear. */
tkg_status tkg_get_device_status(cudaStream_t stream);

/* Static string naming a status code. */
const char *tkg_status_string(tkg_status status);

/* Bytes of a tiled scale buffer for `rows` rows, K = k, block size `block`
 * (32 for MXFP8, 16 for NVFP4): ceil(rows/128)*128 * ceil(ceil(k/block)/4)*4.
 * Returns 0 for invalid arguments. */
size_t tkg_scale_bytes(int rows, int k, int block);

/* Row-major scale matrix (rows x kblocks codes, row pitch ld bytes) -> tiled
 * layout in dst (tkg_scale_bytes(rows, kblocks * block, block) bytes; padding
 * written as zero).  One GPU kernel, byte exact. */
tkg_status tkg_scales_to_tiled(int rows, int kblocks, const void *src, int ld, void *dst, cudaStream_t stream);

/* MXFP8 quantiser, following the workload rule: per 1 x 32 block of each row
 * of X (rows x k FP32, row-major), amax = max |x|, scale exponent
 * e = ceil(log2(amax / 448)) (smallest e with 448 * 2^e >= amax, clamped to
 * [-127, 127]; an all-zero block gets -127), code = e + 127, and
 * q = E4M3 round-to-nearest-even, saturating, of x * 2^-e (FP32).
 * Q: rows x k bytes; sf: tiled layout (bs = 32).  Requires k % 32 == 0. */
tkg_status tkg_quantize_mxfp8(int rows, int k, const float *X, void *Q, void *sf, cudaStream_t stream);

/* NVFP4 quantiser, following the workload rule, every step one FP32 IEEE
 * operation in the order written:
 *   t = amax(X) / 2688 (= 6 * 448);  per 1 x 16 block:
 *   s = E4M3_rne_sat(blockamax / (6 * t));  q = E2M1_rne_sat(x / (dec(s) * t)).
 * t == 0 or dec(s) == 0 gives q = 0.  Q: rows x k/2 bytes (low nibble first),
 * sf: tiled layout (bs = 16), tensor_scale: one FP32 written with t.
 * Requires k % 32 == 0. */
tkg_status tkg_quantize_nvfp4(int rows, int k, const float *X, void *Q, void *sf, float *tensor_scale,
                              cudaStream_t stream);

/* The NVFP4 quantiser with the FP32 tensor scale t supplied instead of
 * computed: the per-block steps above, with t read from tensor_scale (device,
 * one FP32, not written).  For a calibrated or global activation scale, or to
 * quantise slices of one tensor (say each expert's rows of a mixture-of-experts
 * batch, each into its own 128-row scale block) with the scale of the whole.
 * Blocks whose maximum exceeds 6 * 448 * t saturate (scale 448, codes 6);
 * t <= 0 or NaN gives all-zero codes and scales.  Q and sf as above.
 * Errors: tensor_scale NULL -> TKG_ERR_INVALID_ARG, not 4-byte aligned ->
 * TKG_ERR_ALIGNMENT; otherwise as tkg_quantize_nvfp4. */
tkg_status tkg_quantize_nvfp4_scaled(int rows, int k, const float *X, void *Q, void *sf, const float *tensor_scale,
                                     cudaStream_t stream);

/* Process-wide tuning and test options (all default to 0 = automatic). */
typedef enum {
  TKG_OPT_CTA_GROUP = 1,      /* 0 auto, 1 single-CTA MMA, 2 CTA-pair MMA */
  TKG_OPT_SINGLE_STAGE = 2,   /* 1: run the one-stage pipeline build (a test of the ring) */
  TKG_OPT_TIMEOUT_MS = 3,     /* bound on every device wait, milliseconds (0: 1000) */
  TKG_OPT_INJECT_STALL = 4,   /* 1: the MMA role waits on a barrier nothing arrives on
                                  (test of the timeout path; output is garbage) */
  TKG_OPT_MAX_CLUSTERS = 5,   /* cap on persistent clusters (0: fill the GPU) */
  TKG_OPT_ACC_STAGES = 6,     /* BF16 only: 1 = single accumulator buffer (0: double) */
  TKG_OPT_SCHEDULER = 7,      /* 0: cluster launch control (one cluster per tile, running
                                  clusters take over pending ones); 1: static persistent
                                  grid (TKG_OPT_MAX_CLUSTERS applies only here) */
  TKG_OPT_SPLIT_K = 8,        /* 0: split K across 2-3 CTAs when the output has few 128x128
                                  tiles (skinny M) and all their clusters can be resident at
                                  once; 1: never; 2, 3: that split whenever valid */
  TKG_OPT_RASTER_GROUP = 9,   /* M-blocks per tile-order band (0: sized from L2 and K) */
  TKG_OPT_BF16_TILE_N = 10,   /* BF16 CTA-pair tile width: 256 (two accumulator buffers) or
                                  512 (dual accumulate: two N=256 MMAs share each A tile);
                                  0: automatic */
  TKG_OPT_TAIL_SPLIT = 11,    /* plain GEMMs on the persistent kernel: 0 splits the last partial
                                  wave of tiles into half-width tiles when those still fit one
                                  wave; 1 never; 2 splits every tile (a test of the half tiles) */
  TKG_OPT_EPILOGUE_STORE = 12 /* plain GEMMs on the persistent kernel: how the epilogue writes D;
                                  1 TMA stores of 32 x 32 boxes staged in shared memory, 2 16-byte
                                  stores from registers; 0 automatic */
} tkg_option;

tkg_status tkg_set_option(tkg_option option, int value);
int tkg_get_option(tkg_option option);

#ifdef __cplusplus
}
#endif
#endif /* TKG_GEMM_H */
