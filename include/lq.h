/*
 * lq.h -- C ABI of liblq: per-tile randomized Hadamard transform (RHT) plus
 * nearest-point lattice vector quantization of weight matrices, and the
 * products y = W^ x computed straight from the lattice codes, on one
 * sm_103a GPU.
 *
 * Method source: HyperQuant (github release page of moonmath-ai/HyperQuant),
 * sections "Key algorithmic ingredients" (per-tile RHT, E8/D4/A2/Z1 lattice VQ),
 * the mma="int8" paragraph (codes expanded to int8 on chip, the activation
 * rotated at each forward, the weight never materialised in bf16), the
 * mma="bf16" paragraph (the product accumulated from the codes as they are
 * decoded) and "Hadamard block size" (tile rule).
 * Nearest-point algorithms: Conway & Sloane, Sphere Packings, Lattices and
 * Groups, ch. 20.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All matrices are row-major.  W is [rows x cols] (rows = out_features,
 *   cols = in_features).  A tile is a run of `tile` consecutive columns of
 *   one row; `cols % tile == 0`.
 * - Pointers named *_dev are device pointers owned by the caller; the library
 *   never allocates, frees or retains them.  Device pointers must be 16-byte
 *   aligned.  `stream` is a cudaStream_t passed as void* (NULL = legacy
 *   default stream).  Every call only enqueues work on `stream` and returns.
 *   That work is stream-ordered: it reads its inputs after everything
 *   enqueued before it has finished, and what follows it sees its results.
 *   Within a call, and from one product call to the next, kernels are
 *   programmatic dependent launches: a kernel may be scheduled while the one
 *   before it ends, and waits for that grid before it touches data the
 *   earlier work may write.
 * - Argument errors are returned synchronously, before anything is launched.
 *   Data-dependent problems (non-finite input, a code outside int8, a wait
 *   that gave up) are OR-ed as LQ_DEV_* bits into the caller's int32 status
 *   word `dev_status_dev` (may be NULL to ignore them); read it after the
 *   stream has synchronised.  No kernel traps or spins without a bound.
 * - Lattice codes are int8 "doubled coordinates": code = 2 p for a lattice
 *   point p (E8, D4, Z1), and (2x, 2y/sqrt(3)) for an A2 point (x, y).  Codes
 *   are stored [rows x cols], the block of lattice dimension n of tile t at
 *   columns t*tile + n*j ... n*j + n - 1.
 * - Scales are float32 [rows x cols/tile]: s = beta * RMS(tile), the RMS of
 *   the tile before or after the (orthonormal) rotation.
 * - Signs are int8 +1/-1 [cols], one per column, shared by all rows; the
 *   rotation of a tile is w~ = H D w / sqrt(tile) (H Sylvester Hadamard in
 *   natural order, D = diag(signs)).
 */
#ifndef LQ_H
#define LQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Synchronous status returned by every entry point. */
typedef enum {
    LQ_OK = 0,
    LQ_ERR_ARG = 1,         /* null pointer, bad enum value, misaligned pointer */
    LQ_ERR_SHAPE = 2,       /* sizes inconsistent or out of the supported range */
    LQ_ERR_DTYPE = 3,       /* unsupported element type */
    LQ_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, attribute, ...) */
    LQ_ERR_UNSUPPORTED = 5  /* valid request that this library does not implement */
} lq_status;

/* Bits OR-ed into the device status word by the kernels. */
enum {
    LQ_DEV_NONFINITE = 1,   /* a tile held NaN or Inf: that tile's codes are unspecified */
    LQ_DEV_RANGE = 2,       /* some |code| > 127 (or an fp16 activation overflowed) */
    LQ_DEV_TIMEOUT = 4,     /* a bounded wait on an mbarrier expired; outputs unspecified */
    LQ_DEV_FORMAT = 8       /* codes given to the Rice encoder lack the lattice's pinned bits */
};

typedef enum { LQ_Z1 = 1, LQ_A2 = 2, LQ_D4 = 4, LQ_E8 = 8 } lq_lattice;
typedef enum { LQ_F32 = 0, LQ_BF16 = 1 } lq_dtype;

/* Human-readable name of a status code (static string). */
const char* lq_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int lq_version(void);

/*
 * Tile-size rule (HyperQuant page, "Hadamard block size"): the largest tile in
 * {256, 512, 1024, 2048} that is <= `requested` and divides `cols`; 0 when
 * none does.  Pure host function.
 */
int lq_pick_tile(int64_t cols, int requested);

/*
 * Rademacher signs of the RHT (HyperQuant page, "Key algorithmic
 * ingredients": randomized Hadamard).  signs_dev[k] = -1 when the top bit of
 * output k of SplitMix64 started from state `seed` is set (output k mixes
 * seed + (k+1) * 0x9E3779B97F4A7C15), else +1.  signs_dev: int8 [cols].
 */
lq_status lq_make_signs(uint64_t seed, int64_t cols, int8_t* signs_dev, void* stream);

/*
 * Quantize W (HyperQuant page, "Key algorithmic ingredients"; Conway & Sloane
 * ch. 20).  For every tile of every row: sign flip by D, Hadamard, s = beta *
 * RMS, y = w~ / s (s == 0 gives y = 0), nearest lattice point of every
 * n-block of y (E8: the closer of the D8 and D8+1/2 decodes, D8 kept on equal
 * distance; D_n: round, fix parity on the worst coordinate, lowest index on
 * ties; ties of rounding go to even), codes = doubled coordinates.
 *
 *   lattice   LQ_E8 / LQ_D4 / LQ_A2 / LQ_Z1
 *   W_dev     [rows x ldw] elements of type wdtype (LQ_BF16 or LQ_F32);
 *             ldw >= cols and ldw * sizeof(elem) % 16 == 0
 *   tile      128, 256, 512, 1024 or 2048 (cols % tile == 0)
 *   seed      signs are generated from it into signs_dev (int8 [cols], written)
 *   beta      > 0
 *   codes_dev int8 [rows x cols] (written, row stride cols)
 *   scales_dev float32 [rows x cols/tile] (written)
 *   dev_status_dev  int32 status word or NULL (LQ_DEV_NONFINITE, LQ_DEV_RANGE)
 * Limits: rows >= 0, 0 < cols <= 2^20, rows * cols < 2^40.
 */
lq_status lq_quantize(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                      int64_t ldw, int tile, uint64_t seed, float beta,
                      int8_t* codes_dev, float* scales_dev, int8_t* signs_dev,
                      int32_t* dev_status_dev, void* stream);

/*
 * lq_quantize over a group of n matrices (for example the seven linear layers
 * of a transformer block) in one launch pair instead of n.  The pages quantize
 * every linear layer of a model independently; grouping only merges launches:
 * every matrix's signs, codes and scales equal those of lq_quantize with its
 * own arguments.
 *   n          1 .. LQ_QUANTIZE_MAX_GROUP
 *   W_dev, codes_dev, scales_dev, signs_dev
 *              HOST arrays of n DEVICE pointers, one entry per matrix, each as
 *              in lq_quantize
 *   rows, cols, ldw, seeds
 *              HOST arrays of n values, each as in lq_quantize (rows 0
 *              allowed: that matrix only gets its signs)
 *   lattice, wdtype, tile, beta   shared by the group, as in lq_quantize
 *   dev_status_dev  one int32 status word for the whole group, or NULL
 * The host arrays are read during the call only.  Errors as in lq_quantize
 * (the first failing matrix decides, before any launch); LQ_ERR_ARG when n is
 * out of range.  Limit: at most 2^40 warp units of 2048 columns in all.
 */
#define LQ_QUANTIZE_MAX_GROUP 8
lq_status lq_quantize_grouped(int lattice, int n, const void* const* W_dev, int wdtype,
                              const int64_t* rows, const int64_t* cols, const int64_t* ldw, int tile,
                              const uint64_t* seeds, float beta, int8_t* const* codes_dev,
                              float* const* scales_dev, int8_t* const* signs_dev,
                              int32_t* dev_status_dev, void* stream);

/*
 * Reconstruct W^ = D H (s * p) / sqrt(tile) per tile, the inverse of the
 * rotation applied to the scaled lattice points (HyperQuant page, mma="int8"
 * paragraph: the codes are decoded, never stored as a weight).
 *   codes_dev int8 [rows x cols], scales_dev float32 [rows x cols/tile],
 *   signs_dev int8 [cols]; What_dev [rows x cols] of type out_dtype (written).
 */
lq_status lq_dequantize(int lattice, const int8_t* codes_dev, const float* scales_dev,
                        const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                        void* What_dev, int out_dtype, void* stream);

/*
 * Workspace bytes lq_gemv needs for `batch` activation rows of length `cols`
 * with tile `tile` (the rotated activation in fp16 plus one float per
 * (row, tile)).  lq_gemv_grouped_workspace_size(n, ...) is the same
 * for n matrices (one rotated activation per matrix).
 */
size_t lq_gemv_workspace_size(int batch, int64_t cols, int tile);

/*
 * Decode-side product y = W^ x from the codes (HyperQuant page, mma="bf16"
 * paragraph: the product is accumulated from the codes, no decoded weight is
 * stored; mma="int8" paragraph: the activation is rotated at each forward):
 *     y[b, r] = sum_t s[r, t] * sum_i p[r, t, i] * x~[b, t, i],
 *     x~ = H D x / sqrt(tile) per tile.
 *   x_dev     [batch x cols] of type xdtype (LQ_BF16 or LQ_F32), row stride cols
 *   batch     1 .. 16
 *   y_dev     float32 [batch x rows] (overwritten)
 *   workspace_dev  lq_gemv_workspace_size(batch, cols, tile) bytes, 16-byte aligned
 *   dev_status_dev  int32 status word or NULL (LQ_DEV_NONFINITE if an
 *             activation row holds a non-finite value; y is then unspecified)
 * Two kernels run on `stream`: the activation rotation, then the product.
 */
lq_status lq_gemv(int lattice, const int8_t* codes_dev, const float* scales_dev,
                  const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                  const void* x_dev, int xdtype, int batch, float* y_dev,
                  void* workspace_dev, int32_t* dev_status_dev, void* stream);

/*
 * lq_gemv over a group of n matrices that share one activation x (for example
 * the q, k and v projections of a transformer layer, or its gate and up
 * projections), in one launch pair instead of n.  The method's pages describe
 * the product per linear layer; grouping only merges launches: every result
 * equals the lq_gemv of that matrix.
 *   n          1 .. LQ_GEMV_MAX_GROUP
 *   codes_dev, scales_dev, signs_dev, y_dev
 *              HOST arrays of n DEVICE pointers, one entry per matrix, each as
 *              in lq_gemv (matrix m has rows[m] rows, cols columns, its own
 *              signs and scales, and writes y_dev[m], float32 [batch x rows[m]])
 *   rows       HOST array of n row counts (0 allowed: that matrix is skipped)
 *   cols, tile, x_dev, xdtype, batch   shared by the group, as in lq_gemv
 *   workspace_dev  lq_gemv_grouped_workspace_size(n, batch, cols, tile) bytes,
 *             16-byte aligned
 * The host arrays are read during the call only.  Errors as in lq_gemv;
 * LQ_ERR_ARG when n is out of range.
 */
#define LQ_GEMV_MAX_GROUP 8
size_t lq_gemv_grouped_workspace_size(int n, int batch, int64_t cols, int tile);
lq_status lq_gemv_grouped(int lattice, int n, const int8_t* const* codes_dev,
                          const float* const* scales_dev, const int8_t* const* signs_dev,
                          const int64_t* rows, int64_t cols, int tile, const void* x_dev,
                          int xdtype, int batch, float* const* y_dev, void* workspace_dev,
                          int32_t* dev_status_dev, void* stream);

/*
 * lq_gemv without a caller-provided workspace (the method's pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory).  Such callers include inference-engine plug-ins whose host engine
 * owns every device allocation through its own pool and forbids allocation at
 * run time, and latency-critical decode loops where an allocation's implicit
 * device synchronisation is not acceptable.
 *
 * Same arguments and result as lq_gemv minus the workspace.  The workspace is
 * a fixed array of LQ_GEMV_NOALLOC_MAX_WORKSPACE bytes inside the library's
 * device image: every GPU that loads the library holds it until the process
 * exits.  Requests whose lq_gemv_workspace_size(batch, cols, tile) exceeds that
 * size return LQ_ERR_SHAPE before anything is launched: a request fits when
 * align256(batch * cols * 2) + align256(batch * (cols / tile) * 4) <=
 * LQ_GEMV_NOALLOC_MAX_WORKSPACE (align256 rounds up to a multiple of 256), for
 * example batch 16 with cols = 131072 at any tile >= 128.  The first call on a
 * device looks the array's device address up (cudaGetSymbolAddress); make that
 * first call before any stream capture.  The address is looked up again when
 * the device's current context changes (after cudaDeviceReset the array may
 * sit elsewhere); that call too should come before any stream capture.
 * Nothing is allocated by this call.  All calls share the one
 * array, so calls that may overlap on the GPU (different streams without
 * ordering between them) race and must not be issued; calls on one stream are
 * ordered and safe.  The array keeps the previous call's contents; the call
 * rewrites every part it reads.
 */
#define LQ_GEMV_NOALLOC_MAX_WORKSPACE ((size_t)4 * 1024 * 1024 + (size_t)64 * 1024)
lq_status lq_gemv_noalloc(int lattice, const int8_t* codes_dev, const float* scales_dev,
                          const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                          const void* x_dev, int xdtype, int batch, float* y_dev,
                          int32_t* dev_status_dev, void* stream);

/*
 * Workspace bytes lq_gemm needs for an output of type ydtype (LQ_F32 or
 * LQ_BF16): the rotated activations X~ as fp16 [M x K], one float per token
 * row and one per weight row, and for a bf16 output the float32 sums [M x N]
 * that the K splits of the launch add into before the final rounding.
 * 0 for an invalid ydtype or a non-positive size.
 */
size_t lq_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int ydtype);

/*
 * Prefill product Y[M x N] = X W^T from the lattice codes of W [N x K]
 * (HyperQuant page, mma="int8" paragraph: tensor-core GEMM on the decoded
 * codes, the activation rotated on every forward, no decoded weight written
 * to memory, a bf16 result; best for prefill / large batch):
 *     Y[m, n] = sum_t s[n, t] * sum_i p[n, t, i] * X~[m, t, i],
 *     X~ = H D X / sqrt(tile) per tile.
 * On chip the decoded weights p s are formed in fp16 (times a per-row power of
 * two) and X~ is rounded to fp16 (times a per-token-row power of two); the
 * tcgen05 tensor cores accumulate in fp32.
 *   codes_dev int8 [N x K], scales_dev float32 [N x K/tile], signs_dev int8 [K]
 *   X_dev     bf16 [M x K] (raw 16-bit patterns), row stride K
 *   tile      128, 256, 512, 1024 or 2048;  K % tile == 0;  N >= 0 (any; the
 *             last 128-row weight tile may be partial);  M >= 0
 *   Y_dev     [M x N] of type ydtype (overwritten): LQ_F32 (the parity
 *             output) or LQ_BF16 (the page's output type; the float32 result
 *             rounded to nearest even)
 *   workspace_dev  lq_gemm_workspace_size(M, N, K, ydtype) bytes, 256-byte aligned
 *   dev_status_dev  int32 status word or NULL (LQ_DEV_NONFINITE for a
 *             non-finite activation row, LQ_DEV_TIMEOUT if a pipeline wait
 *             gave up -- Y is then unspecified)
 * Two kernels run on `stream` (the activation rotation, then the GEMM), and a
 * third for a bf16 output whose launch splits K across CTAs (the rounding of
 * the float32 sums).  LQ_ERR_DTYPE for another ydtype.
 */
lq_status lq_gemm(int lattice, const int8_t* codes_dev, const float* scales_dev,
                  const int8_t* signs_dev, int64_t N, int64_t K, int tile,
                  const uint16_t* X_dev, int64_t M, void* Y_dev, int ydtype,
                  void* workspace_dev, int32_t* dev_status_dev, void* stream);

/*
 * Self-test of the GEMM's bounded pipeline waits; not part of the method (the
 * pages have no counterpart).  Same arguments and preconditions as lq_gemm,
 * with dev_status_dev required.  It launches lq_gemm's kernel in a variant
 * whose activation (X~) producer never fills its ring and whose waits give up
 * after about 2e5 clock cycles (~0.1 ms) instead of about a second: the MMA
 * issuer's wait for the first X~ tile expires, LQ_DEV_TIMEOUT is OR-ed into
 * *dev_status_dev, the code producer waits for its copies in flight, the tensor
 * memory is released, and the kernel returns.  Y is unspecified afterwards;
 * the context stays usable and later calls on the stream run normally.
 */
lq_status lq_gemm_wait_expiry_test(int lattice, const int8_t* codes_dev, const float* scales_dev,
                                   const int8_t* signs_dev, int64_t N, int64_t K, int tile,
                                   const uint16_t* X_dev, int64_t M, void* Y_dev, int ydtype,
                                   void* workspace_dev, int32_t* dev_status_dev, void* stream);

/*
 * ------------------------------------------------------------------------
 * Rice format of the codes (HyperQuant page, "Key algorithmic ingredients":
 * the bits the lattice fixes are dropped, the rest Rice coded; mma="bf16"
 * paragraph: the weight stored as that ~4 bps stream and read by the GEMV
 * without an int8 copy).  The
 * pages fix no layout; this library's format is:
 *  - per block of n codes: E8 and A2 store the block's common parity as one raw
 *    bit, then the halved codes u_i = floor(c_i / 2); D4 and Z1 codes are even
 *    and store u_i = c_i / 2.  E8 and D4: the u_i sum to an even number, so
 *    the last one is stored as floor(u_{n-1} / 2).
 *  - symbols are zigzag-mapped (z = 2u, or -2u - 1 for u < 0) and Rice coded
 *    with parameter K: floor(z / 2^K) one-bits, a zero-bit, the K low bits of z
 *    (least significant first).
 *  - one segment per (row, tile): K (0..7, the shortest segment, smallest K on
 *    ties) in 3 bits, then the blocks in column order.  Segments follow each
 *    other in row-major (row, tile) order without padding; stream bit b is bit
 *    (b mod 32) of 32-bit word b / 32.  tile_offsets[row * tiles + tile] is the
 *    segment's first bit.
 * Limits: rows * cols <= 2^28 (offsets are 32-bit bit counts).
 * ------------------------------------------------------------------------
 */

/* Bytes a stream may need for these codes (worst case plus 16 bytes of
 * padding); 0 for invalid shapes. */
size_t lq_rice_stream_bound(int lattice, int64_t rows, int64_t cols, int tile);

/* Workspace bytes of lq_rice_encode (segment lengths, K values, scan sums). */
size_t lq_rice_workspace_size(int64_t rows, int64_t cols, int tile);

/*
 * Encode int8 codes [rows x cols] (as written by lq_quantize) into the Rice
 * format.
 *   stream_dev        uint32 words, stream_bytes >= lq_rice_stream_bound(...);
 *                     zeroed, then written; 16-byte aligned
 *   tile_offsets_dev  uint32 [rows x cols/tile] (written)
 *   total_bits_dev    one uint64 (written): the stream's length in bits
 *   workspace_dev     lq_rice_workspace_size(...) bytes, 256-byte aligned
 *   dev_status_dev    LQ_DEV_FORMAT when a block lacks the pinned bits (its
 *                     segment then does not decode to the same codes)
 * Six kernels run on `stream` (lengths, three scan passes, bits).
 */
lq_status lq_rice_encode(int lattice, const int8_t* codes_dev, int64_t rows, int64_t cols, int tile,
                         uint32_t* stream_dev, size_t stream_bytes, uint32_t* tile_offsets_dev,
                         uint64_t* total_bits_dev, void* workspace_dev, int32_t* dev_status_dev,
                         void* stream);

/*
 * Decode a Rice stream back into int8 codes [rows x cols] (written).  Reads
 * never go past stream_bytes (bits beyond it read as zero).
 */
lq_status lq_rice_decode(int lattice, const uint32_t* stream_dev, size_t stream_bytes,
                         const uint32_t* tile_offsets_dev, int64_t rows, int64_t cols, int tile,
                         int8_t* codes_dev, void* stream);

/*
 * lq_gemv computed from the Rice stream instead of int8 codes: the codes are
 * decoded inside the product (never written to memory).  Arguments as in
 * lq_gemv, with (stream_dev, stream_bytes, tile_offsets_dev) in place of
 * codes_dev; workspace_dev has lq_gemv_workspace_size(batch, cols, tile) bytes.
 */
lq_status lq_gemv_rice(int lattice, const uint32_t* stream_dev, size_t stream_bytes,
                       const uint32_t* tile_offsets_dev, const float* scales_dev,
                       const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                       const void* x_dev, int xdtype, int batch, float* y_dev, void* workspace_dev,
                       int32_t* dev_status_dev, void* stream);

/*
 * ------------------------------------------------------------------------
 * Rate / SNR calibration (HyperQuant page, usage section and "bps" table: rates
 * in bits per scalar are related to SNRs by measurement, and the lattice
 * scale is set from a target SNR).  SNR = 10 log10(sum w^2 /
 * sum (w - w^)^2) in dB.
 * ------------------------------------------------------------------------
 */

/* beta giving `snr_db` in the high-resolution regime: sqrt(10^(-snr/10) /
 * (G V^(2/n))), G the lattice's normalised second moment (Conway & Sloane
 * table 2.3), V its cell volume at the quantizer's scale.  Host only; 0 for an
 * invalid lattice. */
double lq_beta_for_snr(int lattice, double snr_db);

/* sums_dev[0] = sum w^2, sums_dev[1] = sum (w - w^)^2 (double; zeroed first)
 * over W [rows x ldw] (bf16 or fp32) and W^ float32 [rows x cols]. */
lq_status lq_error_sums(const void* W_dev, int wdtype, int64_t rows, int64_t cols, int64_t ldw,
                        const float* What_dev, double* sums_dev, void* stream);

/* Workspace bytes of lq_calibrate_bps (codes, scales, signs, Rice stream and
 * its workspace, a float32 reconstruction); 0 for unsupported shapes. */
size_t lq_calibrate_workspace_size(int lattice, int64_t rows, int64_t cols, int tile);

/*
 * The scale beta at which the Rice rate of the sample W (bits per weight of
 * the bit-stripped stream) is at most `target_bps`: bisection on log2(beta)
 * over [-8, 4], 24 halvings, keeping the upper end; each probe quantizes
 * (signs from `seed`) and encodes on the GPU, and a probe whose codes leave
 * int8 counts as above the target.  SYNCHRONOUS: returns after the
 * stream has drained.  result (host, 3 doubles) = {beta, bits per weight,
 * SNR in dB} at that beta.  LQ_ERR_UNSUPPORTED when the final scale leaves
 * int8 (targets above about 6 bps) or the sample is not finite.
 */
lq_status lq_calibrate_bps(int lattice, int tile, double target_bps, const void* W_dev, int wdtype,
                           int64_t rows, int64_t cols, int64_t ldw, uint64_t seed, void* workspace_dev,
                           size_t workspace_bytes, double* result, void* stream);

/*
 * ------------------------------------------------------------------------
 * KV cache (HyperQuant page, KV-cache section: lattice codes plus one norm per
 * vector after a random sign rotation; attention on the quantized cache).  A
 * K or V cache [tokens x kv_heads * head_dim] is quantized with lq_quantize,
 * tile = head_dim: every (token, head) vector is one tile, its scale the
 * vector's norm / sqrt(head_dim) * beta.
 * ------------------------------------------------------------------------
 */

/* Workspace bytes of lq_attention_decode; 0 for unsupported shapes. */
size_t lq_attention_workspace_size(int64_t tokens, int kv_heads, int q_heads, int head_dim);

/*
 * One decode step of attention over quantized K and V caches, computed from
 * the codes (no dequantized cache in memory):
 *     out[h] = softmax(K^_g q[h] / sqrt(head_dim)) V^_g,  g = h / (q_heads / kv_heads)
 *   k_codes_dev, v_codes_dev   int8 [tokens x kv_heads * head_dim]
 *   k_scales_dev, v_scales_dev float32 [tokens x kv_heads]
 *   k_signs_dev, v_signs_dev   int8 [kv_heads * head_dim]
 *   q_dev      [q_heads x head_dim] of type qdtype (LQ_BF16 or LQ_F32)
 *   out_dev    float32 [q_heads x head_dim] (written)
 *   head_dim   128;  q_heads / kv_heads in {1, 2, 4, 8};  tokens >= 1
 *   workspace_dev  lq_attention_workspace_size(...) bytes (workspace_bytes)
 * Two kernels run on `stream` (per-range partial softmax sums, then the merge
 * and the inverse rotation).
 */
lq_status lq_attention_decode(int lattice, const int8_t* k_codes_dev, const float* k_scales_dev,
                              const int8_t* k_signs_dev, const int8_t* v_codes_dev,
                              const float* v_scales_dev, const int8_t* v_signs_dev, int64_t tokens,
                              int kv_heads, int q_heads, int head_dim, const void* q_dev, int qdtype,
                              float* out_dev, void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * The "qjl" rotation of the KV cache (HyperQuant page, KV-cache section:
 * Haar-uniform rotation for unbiased inner products): y = M x for every
 * head_dim-column block x of every row of X, M = R (transpose = 0) or R^T
 * (transpose = 1).  R_dev: float32 [head_dim x head_dim] row-major, an
 * orthogonal matrix drawn by the caller; X [rows x ldx] bf16 or fp32; Y float32
 * [rows x ldy] (written).  Rotate K/V rows and queries by R before quantizing /
 * attending, and the attention output back by R^T.  head_dim 128.
 */
lq_status lq_rotate_blocks(const float* R_dev, int transpose, int head_dim, const void* X_dev,
                           int xdtype, int64_t rows, int64_t cols, int64_t ldx, float* Y_dev,
                           int64_t ldy, void* stream);

/*
 * ------------------------------------------------------------------------
 * Scale formats.  Every call above stores and reads one float32 scale per
 * (row, tile).  The _ex calls below take the format as an argument:
 *   LQ_SCALE_TILE_F32  float32 [rows x cols/tile]: the format of the calls above.
 *   LQ_SCALE_ROW_BF16  bfloat16 [rows] (raw 16-bit patterns): one scale per row,
 *                      s_r = beta * RMS of the whole row (HyperQuant page,
 *                      mma="int8" paragraph: each output row normalised by
 *                      its own statistic, one bf16 scale stored per row).
 *   LQ_SCALE_TILE_F16  float16 [rows x cols/tile] (raw 16-bit patterns): the
 *                      per-tile scale in half precision (the page's KV cache:
 *                      int8 codes with fp16 norms).
 * With a 16-bit format the stored value is the scale rounded to nearest-even,
 * and the codes are the nearest lattice points of the rotated tile divided by
 * that stored value, so that reconstruction and products use exactly what is
 * stored.  An fp16 scale that overflows raises LQ_DEV_RANGE (codes of that tile
 * unspecified); a row holding a non-finite value gets scale 0 and
 * LQ_DEV_NONFINITE.
 * ------------------------------------------------------------------------
 */
#define LQ_SCALE_TILE_F32 0
#define LQ_SCALE_ROW_BF16 1
#define LQ_SCALE_TILE_F16 2

/* lq_quantize writing scales_dev in scale_format.  LQ_SCALE_ROW_BF16 reads W
 * twice (a row-norm pass, then the quantize pass), in row blocks small enough
 * for the second read to come from L2. */
lq_status lq_quantize_ex(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                         int64_t ldw, int tile, uint64_t seed, float beta, int scale_format,
                         int8_t* codes_dev, void* scales_dev, int8_t* signs_dev,
                         int32_t* dev_status_dev, void* stream);

/* lq_dequantize reading scales_dev in scale_format. */
lq_status lq_dequantize_ex(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                           const int8_t* signs_dev, int64_t rows, int64_t cols, int tile, void* What_dev,
                           int out_dtype, void* stream);

/* lq_gemv reading scales_dev in scale_format (same workspace). */
lq_status lq_gemv_ex(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                     const int8_t* signs_dev, int64_t rows, int64_t cols, int tile, const void* x_dev,
                     int xdtype, int batch, float* y_dev, void* workspace_dev, int32_t* dev_status_dev,
                     void* stream);

/* lq_gemm reading scales_dev in scale_format (same workspace and output types). */
lq_status lq_gemm_ex(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                     const int8_t* signs_dev, int64_t N, int64_t K, int tile, const uint16_t* X_dev, int64_t M,
                     void* Y_dev, int ydtype, void* workspace_dev, int32_t* dev_status_dev, void* stream);

/* lq_attention_decode with both caches' scales in scale_format
 * (LQ_SCALE_TILE_F32 or LQ_SCALE_TILE_F16, [tokens x kv_heads]). */
lq_status lq_attention_decode_ex(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                                 const int8_t* k_signs_dev, const int8_t* v_codes_dev, const void* v_scales_dev,
                                 const int8_t* v_signs_dev, int scale_format, int64_t tokens, int kv_heads,
                                 int q_heads, int head_dim, const void* q_dev, int qdtype, float* out_dev,
                                 void* workspace_dev, size_t workspace_bytes, void* stream);

/*
 * ------------------------------------------------------------------------
 * Subtractive Voronoi dither (HyperQuant page, "Key algorithmic ingredients":
 * one of two listed ways to keep the cache's inner products unbiased; Zamir &
 * Feder, "On lattice quantization noise", 1996: the reconstruction error is
 * then uniform over the lattice cell and independent of the input).
 * Element (r, k) of a [rows x cols] matrix draws w = (top 24 bits of SplitMix64
 * output r * cols + k from state dither_seed) / 2^24; the draws of one lattice
 * block, scaled to a box that tiles space under a sublattice (E8, D4: side 2;
 * A2: 1 x sqrt 3; Z1: 1), are reduced into the Voronoi cell: u = z - Q(z).
 * The codes are those of Q(y + u), y the scaled rotated tile; the reconstruction
 * is s (p - u).  Codes and scales keep their layouts; scale_format is
 * LQ_SCALE_TILE_F32 or LQ_SCALE_TILE_F16.  A tile with a zero scale keeps zero
 * codes (no dither).
 * ------------------------------------------------------------------------
 */
lq_status lq_quantize_dithered(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                               int64_t ldw, int tile, uint64_t seed, uint64_t dither_seed, float beta,
                               int scale_format, int8_t* codes_dev, void* scales_dev, int8_t* signs_dev,
                               int32_t* dev_status_dev, void* stream);

/* W^ = D H (s (p - u)) / sqrt(tile) for codes made by lq_quantize_dithered. */
lq_status lq_dequantize_dithered(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                                 const int8_t* signs_dev, uint64_t dither_seed, int64_t rows, int64_t cols,
                                 int tile, void* What_dev, int out_dtype, void* stream);

/* lq_attention_decode_ex over K and V caches made by lq_quantize_dithered with
 * the given dither seeds (K^ = s (p - u) row by row, the same for V^); the
 * dither draws are regenerated on chip, never stored. */
lq_status lq_attention_decode_dithered(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                                       const int8_t* k_signs_dev, uint64_t k_dither_seed,
                                       const int8_t* v_codes_dev, const void* v_scales_dev,
                                       const int8_t* v_signs_dev, uint64_t v_dither_seed, int scale_format,
                                       int64_t tokens, int kv_heads, int q_heads, int head_dim, const void* q_dev,
                                       int qdtype, float* out_dev, void* workspace_dev, size_t workspace_bytes,
                                       void* stream);

/*
 * Decode attention over K and V caches held as Rice streams (HyperQuant page,
 * KV-cache storage table: "Rice bitstream + fp16 norms", ~3.8x against bf16):
 * each cache [tokens x kv_heads * head_dim] is quantized (lq_quantize_ex, tile
 * = head_dim) and then coded with lq_rice_encode (rows = tokens, cols =
 * kv_heads * head_dim, tile = head_dim), one segment per (token, kv head).  The
 * kernel decodes every token's segments on chip and computes what
 * lq_attention_decode_ex computes on the int8 codes.
 *   k_stream_dev / v_stream_dev   the Rice words (k_stream_bytes, v_stream_bytes)
 *   k_offsets_dev / v_offsets_dev uint32 [tokens x kv_heads] segment bit offsets
 *   scales, signs, q, out, workspace, shapes: as in lq_attention_decode_ex
 * At most 2^28 cached values per stream (the format's 32-bit bit offsets).
 */
lq_status lq_attention_decode_rice(int lattice, const uint32_t* k_stream_dev, size_t k_stream_bytes,
                                   const uint32_t* k_offsets_dev, const void* k_scales_dev,
                                   const int8_t* k_signs_dev, const uint32_t* v_stream_dev, size_t v_stream_bytes,
                                   const uint32_t* v_offsets_dev, const void* v_scales_dev,
                                   const int8_t* v_signs_dev, int scale_format, int64_t tokens, int kv_heads,
                                   int q_heads, int head_dim, const void* q_dev, int qdtype, float* out_dev,
                                   void* workspace_dev, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LQ_H */
