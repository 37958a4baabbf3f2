/*
 * taco.h -- C ABI of libtaco_gb300.so: TACO's fused FP8 compression of
 * tensor-parallel intermediate tensors, as CUDA kernels for GB300 (sm_103a).
 *
 * Method: "TACO: Efficient Communication Compression of Intermediate Tensors
 * for Scalable Tensor-Parallel LLM Training", Algorithm 1 and Eqs. (5)-(13),
 * Sections 4.2-4.4.
 *
 * Constants the paper leaves open, fixed here:
 *   tau = 1 (target RMS of a block after the Adaptive Scale, Eq. 7),
 *   eps = 1e-30 (inside the square root of Eq. 6),
 *   Q_max = 448 (largest finite OCP E4M3 value, Eq. 9),
 *   H_B = Sylvester Hadamard matrix in natural order, (H_B)_ij = (-1)^popcount(i&j),
 *   Cvt_FP8 = round to nearest even, saturating to +-448 (Eq. 10).
 *
 * Tensor layout: a row-major bf16 tensor [rows, hidden] with hidden % block == 0,
 * seen as M = rows*hidden/block contiguous blocks of `block` elements (Eq. 5).
 *
 * Packed layout (Section 4.4.2, the codes with their scales stored right
 * after them in the same buffer): one buffer of
 * M records; record k starts at byte k*(block+8) and holds the block's `block`
 * E4M3 codes in element order, then alpha_k and s_k as little-endian float32.
 * taco_compressed_bytes() gives its size.
 *
 * Common rules for every call below:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     16-byte aligned (TACO_ERR_MISALIGNED otherwise).  The caller allocates
 *     and frees every buffer; the library allocates no memory.
 *   - Inputs and outputs must not overlap (TACO_ERR_OVERLAP).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.  TACO_OK means the
 *     kernel was launched.  Argument errors are found on the host before any
 *     launch and leave every output untouched.  Calls keep no state between
 *     them, so calls on different streams (or threads) may run at the same
 *     time on disjoint buffers; within a stream each kernel starts while the
 *     previous one drains but reads its input only once that kernel is done.
 *     The first call on a device does the library's one-time set-up for it
 *     (kernel attributes, the fault flag's address); after that,
 *     taco_compress, taco_decompress and taco_reduce_shards (and their _ex
 *     forms) may be captured into CUDA graphs.  taco_device_status copies
 *     synchronously and is not capturable.
 *   - rows == 0 or hidden == 0 is an empty tensor: TACO_OK, nothing launched,
 *     pointers may be NULL.
 *   - Supported blocks: 32, 64, 128, 256, 512 (TACO_ERR_UNSUPPORTED_BLOCK
 *     otherwise; Section 5.3.3 ablates these sizes).  64 to 512 run on the
 *     tensor cores, 32 on a lane-per-block CUDA-core codec.
 *   - Inputs must be finite with |x| < 2^56; beyond that the FP32 block
 *     energy of Eq. (6) can overflow and the output is unspecified.
 *   - Kernels that wait on the copy engine give up after about one second,
 *     set a device-side fault flag and return; taco_device_status() reads it.
 */
#ifndef TACO_GB300_H
#define TACO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TACO_API __attribute__((visibility("default")))
#else
#define TACO_API
#endif

/* Same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *taco_stream_t;

typedef enum taco_status {
    TACO_OK = 0,
    TACO_ERR_NULL_POINTER = 1,      /* a required pointer is NULL */
    TACO_ERR_BAD_SHAPE = 2,         /* rows < 0, hidden < 0, hidden % block != 0, size overflow, or
                                       (compress / decompress, blocks 64-512) more than 2^31 - 1 rows
                                       of min(block, 128) elements */
    TACO_ERR_UNSUPPORTED_BLOCK = 3, /* block not in {32, 64, 128, 256, 512} */
    TACO_ERR_MISALIGNED = 4,        /* a device pointer is not 16-byte aligned */
    TACO_ERR_BAD_SHARDS = 5,        /* num_shards < 1 or > TACO_MAX_SHARDS */
    TACO_ERR_OVERLAP = 6,           /* an output overlaps an input */
    TACO_ERR_CUDA = 7,              /* a CUDA runtime call or launch failed; see taco_last_cuda_error() */
    TACO_ERR_DEVICE_FAULT = 8,      /* taco_device_status(): a kernel gave up waiting */
    TACO_ERR_BAD_OPTIONS = 9        /* the _ex calls: options NULL, or unknown variant or code format */
} taco_status_t;

#define TACO_MAX_SHARDS 16
#define TACO_ABI_VERSION 2

/*
 * Ablations of the method for the _ex calls (paper Sections 5.2.2, 5.3.1,
 * 5.3.2 and 6).  The record layout is always [block codes | alpha | s].
 */
typedef enum taco_variant {
    TACO_VARIANT_ASH_DS = 0,      /* the method: Adaptive Scale + Hadamard + Dual-Scale */
    TACO_VARIANT_HADAMARD_DS = 1, /* standard Hadamard + Dual-Scale: alpha = 1 (Section 5.3.1) */
    TACO_VARIANT_DS_ONLY = 2,     /* Dual-Scale only: alpha = 1, no rotation (Section 5.2.2) */
    TACO_VARIANT_ASH_ONLY = 3     /* ASH only: s = 1, Z cast directly (Section 5.2.2) */
} taco_variant_t;

typedef enum taco_code {
    TACO_CODE_E4M3 = 0,           /* OCP E4M3FN, Q_max = 448: the method */
    TACO_CODE_E5M2 = 1,           /* OCP E5M2, Q_max = 57344, nearest even, saturating (Section 5.3.2) */
    TACO_CODE_INT8 = 2            /* int8, Q_max = 127, nearest integer with ties to even (Sections 2, 6) */
} taco_code_t;

typedef struct taco_options {
    int block;                    /* 32, 64, 128, 256 or 512 */
    int variant;                  /* taco_variant_t */
    int code;                     /* taco_code_t */
} taco_options_t;

/* Bytes of the packed buffer for a [rows, hidden] tensor: (rows*hidden/block)*(block+8).
 * Returns -1 for an unsupported block, a bad shape or an overflow. */
TACO_API int64_t taco_compressed_bytes(int64_t rows, int64_t hidden, int block);

/*
 * Sender side, Algorithm 1's compression loop (Eqs. 5-10), one fused kernel: for every
 * block G_k of x, sigma_k = sqrt(mean(G_k^2) + eps) (Eq. 6), alpha_k = tau/sigma_k
 * (Eq. 7), Z_k = (1/sqrt B) H_B (alpha_k G_k) (Eq. 8), s_k = max|Z_k| / Q_max
 * (Eq. 9), q_k = Cvt_FP8(Z_k / s_k) (Eq. 10); writes the record (q_k, alpha_k, s_k).
 * A block with max|Z_k| = 0 gets s_k = 0 and all codes 0x00.
 *
 *   x_bf16      device, in:  rows*hidden bf16 values, row-major
 *   packed_out  device, out: taco_compressed_bytes(rows, hidden, block) bytes
 */
TACO_API taco_status_t taco_compress(const void *x_bf16, int64_t rows, int64_t hidden, int block,
                            void *packed_out, taco_stream_t stream);

/*
 * Receiver side, Algorithm 1's decompression loop (Eqs. 11-13), the fused decompress
 * kernel (Section 4.1, "fused_ash_decompress_kernel"): Zhat_k = Cvt_FP32(q_k) s_k,
 * Ghat_k = (1/sqrt B) H_B Zhat_k, G'_k = Ghat_k / alpha_k, rounded to bf16
 * (nearest even).
 *
 *   packed_in   device, in:  taco_compressed_bytes(rows, hidden, block) bytes
 *   y_bf16_out  device, out: rows*hidden bf16 values, row-major
 */
TACO_API taco_status_t taco_decompress(const void *packed_in, int64_t rows, int64_t hidden, int block,
                              void *y_bf16_out, taco_stream_t stream);

/*
 * Receive-side local reduction of the two-shot compressed AllReduce (Section
 * 4.4.2: after the compressed all-to-all exchange, each owner reduces its
 * segment once): the P packed shards of the same [rows, hidden] tensor are
 * decoded to FP32 (Eqs. 11-13, no bf16 rounding), summed, and the FP32 sum is
 * compressed once (Eqs. 6-10) into packed_out.
 *
 *   packed_shards  HOST array of num_shards DEVICE pointers, each to
 *                  taco_compressed_bytes(rows, hidden, block) bytes; the array
 *                  is read during the call only and may be freed afterwards
 *   num_shards     P, 1 <= P <= TACO_MAX_SHARDS
 *   packed_out     device, out: taco_compressed_bytes(rows, hidden, block) bytes,
 *                  overlapping no shard
 */
TACO_API taco_status_t taco_reduce_shards(const void *const *packed_shards, int num_shards, int64_t rows,
                                 int64_t hidden, int block, void *packed_out, taco_stream_t stream);

/*
 * The three calls above for any variant and code format (taco_options_t; the
 * plain calls are block = options->block, TACO_VARIANT_ASH_DS, TACO_CODE_E4M3).
 * Per block, with y the Hadamard rotation H_B G (G itself for DS only), Z =
 * alpha y / sqrt(B) and Q_max of the code format:
 *   ASH + DS            alpha = tau / sigma, s = max|Z| / Q_max, q = Cvt(Z / s)
 *   standard Hadamard   alpha = 1,           s = max|Z| / Q_max, q = Cvt(Z / s)
 *   DS only             alpha = 1, Z = G,    s = max|G| / Q_max, q = Cvt(G / s)
 *   ASH only            alpha = tau / sigma, s = 1,              q = Cvt(Z)
 * and decompression computes (Cvt^-1(q) s, rotated back unless DS only) / alpha.
 * A record must be decoded and reduced with the options it was written with.
 * options == NULL or an unknown variant or code: TACO_ERR_BAD_OPTIONS.
 */
TACO_API taco_status_t taco_compress_ex(const void *x_bf16, int64_t rows, int64_t hidden,
                                        const taco_options_t *options, void *packed_out, taco_stream_t stream);
TACO_API taco_status_t taco_decompress_ex(const void *packed_in, int64_t rows, int64_t hidden,
                                          const taco_options_t *options, void *y_bf16_out, taco_stream_t stream);
TACO_API taco_status_t taco_reduce_shards_ex(const void *const *packed_shards, int num_shards, int64_t rows,
                                             int64_t hidden, const taco_options_t *options, void *packed_out,
                                             taco_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's fault
 * flags (bit 0: compress, bit 1: decompress, bit 2: shard reduce gave up
 * waiting for a copy or a tile assignment; bit 3: the self-test below).
 * *flags_out (may be NULL) receives them.  Returns TACO_ERR_DEVICE_FAULT if any
 * flag was set, TACO_ERR_CUDA if a CUDA call failed, TACO_OK otherwise.
 */
TACO_API taco_status_t taco_device_status(taco_stream_t stream, uint32_t *flags_out);

/*
 * Self-test of the fault path (no counterpart in the paper): launches one CTA
 * on `stream` whose bounded wait on an mbarrier that nothing completes runs
 * out after about 2 ms; it then sets bit 3 of the device fault flags and
 * exits, exactly as every kernel does when a wait gives up.  A following
 * taco_device_status() returns TACO_ERR_DEVICE_FAULT with that bit (and
 * clears it).  Nothing faults, traps or hangs.  Returns TACO_OK once launched.
 */
TACO_API taco_status_t taco_selftest_wait_timeout(taco_stream_t stream);

/*
 * Self-test of the code conversion (no counterpart in the paper): writes
 * codes_out[i] = the code (taco_code_t `code`) of the float32 whose bit
 * pattern is first + i (modulo 2^32), for i < count, computed with the same
 * device function the kernels use to quantize, so that it can be compared with
 * an independent encoder over every float32.  E4M3 and E5M2 use the hardware's
 * saturating round-to-nearest-even conversions (NaN inputs give NaN codes);
 * INT8 rounds half to even and is defined for |u| < 127.5 (the kernels feed
 * it |u| <= 127 up to FP32 rounding).
 *
 *   code       TACO_CODE_E4M3, _E5M2 or _INT8 (TACO_ERR_BAD_OPTIONS otherwise)
 *   first      first bit pattern, a multiple of 4
 *   count      number of codes, a multiple of 4, at most 2^32
 *              (TACO_ERR_BAD_SHAPE otherwise; 0 launches nothing)
 *   codes_out  device, out: count bytes, 16-byte aligned
 */
TACO_API taco_status_t taco_selftest_encode_bits(int code, uint32_t first, int64_t count, void *codes_out,
                                                 taco_stream_t stream);

/* Static, human-readable name of a status. */
TACO_API const char *taco_status_string(taco_status_t status);

/* The cudaError_t value behind the calling thread's last TACO_ERR_CUDA (0 if none). */
TACO_API int taco_last_cuda_error(void);

/* TACO_ABI_VERSION of the loaded library. */
TACO_API int taco_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TACO_GB300_H */
