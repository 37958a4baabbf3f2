// taco_api.cu -- the C ABI of libtaco_gb300.so (declared in include/taco.h):
// argument validation, per-device set-up, grid sizing and kernel launches.
#include <climits>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "taco.h"
#include "taco_kernels.h"

namespace taco {
namespace {

// Device-side fault flags (bits kFaultCompress, kFaultDecompress, kFaultReduce).
__device__ uint32_t g_fault_flags;

thread_local int t_last_cuda_error = 0;

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    int sm_count = 0;
    uint32_t *fault = nullptr;  // device address of g_fault_flags
    int ctas_per_sm = 0;        // last occupancy query (set-up check only)
};

DeviceState g_devices[kMaxDevices];

bool block_supported(int block)
{
    return block == 32 || block == 64 || block == 128 || block == 256 || block == 512;
}

// Blocks 64 .. 512 run on the tensor-core kernels (512 as four rows of 128
// elements per block), 32 on the lane-per-block codec; the shard reduce takes
// every block size.
bool tensor_core_block(int block)
{
    return block == 64 || block == 128 || block == 256 || block == 512;
}

// Row length of the tensor-core kernels' view of the tensor: the block, or
// 128 for B = 256 and 512 (two or four rows per block).
int view_row_elems(int block)
{
    return block > 128 ? 128 : block;
}

taco_status_t cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return TACO_ERR_CUDA;
}

cudaError_t init_kernel(const KernelInfo &ki, int *ctas_per_sm)
{
    cudaError_t e = cudaSuccess;
    if (ki.smem > 48 * 1024)
        e = cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ki.smem));
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, ki.fn, ki.threads, ki.smem);
}

void init_device(DeviceState &st)
{
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&st.fault), g_fault_flags);
    int dev = 0;
    if (e == cudaSuccess)
        e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
    const int blocks[5] = {32, 64, 128, 256, 512};
    for (int i = 0; i < 5 && e == cudaSuccess; i++) {
        if (tensor_core_block(blocks[i])) {
            e = init_kernel(compress_kernel_info(blocks[i], 0, 0), &st.ctas_per_sm);
            if (e == cudaSuccess)
                e = init_kernel(compress_kernel_info(blocks[i], 2, 0), &st.ctas_per_sm);
            if (e == cudaSuccess)
                e = init_kernel(compress_kernel_info(blocks[i], 0, 2), &st.ctas_per_sm);
            for (int code = 0; code < 3 && e == cudaSuccess; code += 2)   // E5M2 shares the E4M3 kernel
                e = init_kernel(decompress_kernel_info(blocks[i], code), &st.ctas_per_sm);
        } else {
            e = init_kernel(warp_codec_info(blocks[i], true, 0), &st.ctas_per_sm);
            if (e == cudaSuccess)
                e = init_kernel(warp_codec_info(blocks[i], true, 2), &st.ctas_per_sm);
            if (e == cudaSuccess)
                e = init_kernel(warp_codec_info(blocks[i], false, 0), &st.ctas_per_sm);
        }
        const int reduce_shards[6] = {1, 2, 4, 5, 8, 16};   // every reduce kernel: generic up to 4, 2, 4, generic, 8, 16
        for (int code = 0; code < 3 && e == cudaSuccess; code++)
            for (int k = 0; k < 6 && e == cudaSuccess; k++)
                e = init_kernel(reduce_kernel_info(blocks[i], code, reduce_shards[k]), &st.ctas_per_sm);
    }
    st.init_error = e;
}

// Set-up of the current device, once per device and process.
taco_status_t device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices)
        return cuda_fail(cudaErrorInvalidDevice);
    DeviceState &st = g_devices[dev];
    std::call_once(st.once, init_device, std::ref(st));
    if (st.init_error != cudaSuccess)
        return cuda_fail(st.init_error);
    *out = &st;
    return TACO_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_error = cudaSuccess;

cudaError_t tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_error = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (g_encode_error == cudaSuccess && (q != cudaDriverEntryPointSuccess || !fn))
            g_encode_error = cudaErrorSymbolNotFound;
        g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    *out = g_encode_tiled;
    return g_encode_error;
}

// Tensor map of a bf16 tensor as [nblocks, block] rows, box {64 elements,
// box_rows rows}, 128-byte swizzle; loads past the end read zeros, stores past
// the end are dropped.
cudaError_t encode_block_rows_map(CUtensorMap *map, const void *x, int64_t nblocks, int block, int box_rows = 128)
{
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaError_t e = tensor_map_encoder(&encode);
    if (e != cudaSuccess)
        return e;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(block), static_cast<cuuint64_t>(nblocks)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(block) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// Validates block and shape; on success sets the element count and packed bytes.
taco_status_t check_shape(int64_t rows, int64_t hidden, int block, int64_t *n, int64_t *packed_bytes)
{
    if (!block_supported(block))
        return TACO_ERR_UNSUPPORTED_BLOCK;
    if (rows < 0 || hidden < 0 || hidden % block != 0)
        return TACO_ERR_BAD_SHAPE;
    if (rows != 0 && hidden > INT64_MAX / 4 / rows)  // keeps 2*n and the packed size in range
        return TACO_ERR_BAD_SHAPE;
    *n = rows * hidden;
    *packed_bytes = *n / block * (block + 8);
    return TACO_OK;
}

// The tensor-core kernels address a tensor as rows of view_row_elems(block)
// elements with 32-bit TMA coordinates: at most INT32_MAX such rows.
taco_status_t check_view_rows(int64_t n, int block)
{
    return tensor_core_block(block) && n / view_row_elems(block) > INT32_MAX ? TACO_ERR_BAD_SHAPE : TACO_OK;
}

taco_status_t check_options(const taco_options_t *opt, Scheme *scheme)
{
    if (!opt)
        return TACO_ERR_BAD_OPTIONS;
    if (opt->variant < TACO_VARIANT_ASH_DS || opt->variant > TACO_VARIANT_ASH_ONLY || opt->code < TACO_CODE_E4M3 ||
        opt->code > TACO_CODE_INT8)
        return TACO_ERR_BAD_OPTIONS;
    *scheme = Scheme{opt->variant, opt->code};
    return TACO_OK;
}

taco_status_t compress_impl(const void *x_bf16, int64_t rows, int64_t hidden, int block, Scheme scheme,
                            void *packed_out, taco_stream_t stream)
{
    int64_t n = 0, bytes = 0;
    taco_status_t st = check_shape(rows, hidden, block, &n, &bytes);
    if (st == TACO_OK)
        st = check_view_rows(n, block);
    if (st != TACO_OK || n == 0)
        return st;
    if (!x_bf16 || !packed_out)
        return TACO_ERR_NULL_POINTER;
    if (!aligned16(x_bf16) || !aligned16(packed_out))
        return TACO_ERR_MISALIGNED;
    if (overlap(x_bf16, 2 * n, packed_out, bytes))
        return TACO_ERR_OVERLAP;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != TACO_OK)
        return st;
    const int64_t nblocks = n / block;
    if (!tensor_core_block(block)) {
        const KernelInfo wk = warp_codec_info(block, true, scheme.code);
        const int64_t want = (nblocks + wk.tile_blocks - 1) / wk.tile_blocks;
        const int64_t cap = static_cast<int64_t>(dev->sm_count) * 16;
        const cudaError_t e = launch_warp_compress(block, scheme, x_bf16, packed_out, nblocks,
                                                   static_cast<int>(want < cap ? want : cap),
                                                   reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? TACO_OK : cuda_fail(e);
    }
    // Tensor-core kernel over tiles of 128 blocks: one CTA per tile, of which
    // one per SM runs and takes the tiles of CTAs it cancels before they start.
    const KernelInfo ki = compress_kernel_info(block, scheme.variant, scheme.code);
    const int64_t ntiles = (nblocks + ki.tile_blocks - 1) / ki.tile_blocks;
    if (ntiles > INT32_MAX)
        return TACO_ERR_BAD_SHAPE;
    alignas(64) CUtensorMap map;
    const int re = view_row_elems(block);
    cudaError_t e = encode_block_rows_map(&map, x_bf16, nblocks * (block / re), re);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const int grid = static_cast<int>(ntiles);
    e = launch_compress(block, scheme, &map, packed_out, nblocks, dev->fault, grid,
                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TACO_OK : cuda_fail(e);
}

taco_status_t decompress_impl(const void *packed_in, int64_t rows, int64_t hidden, int block, Scheme scheme,
                              void *y_bf16_out, taco_stream_t stream)
{
    int64_t n = 0, bytes = 0;
    taco_status_t st = check_shape(rows, hidden, block, &n, &bytes);
    if (st == TACO_OK)
        st = check_view_rows(n, block);
    if (st != TACO_OK || n == 0)
        return st;
    if (!packed_in || !y_bf16_out)
        return TACO_ERR_NULL_POINTER;
    if (!aligned16(packed_in) || !aligned16(y_bf16_out))
        return TACO_ERR_MISALIGNED;
    if (overlap(packed_in, bytes, y_bf16_out, 2 * n))
        return TACO_ERR_OVERLAP;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != TACO_OK)
        return st;
    const int64_t nblocks = n / block;
    if (!tensor_core_block(block)) {
        const KernelInfo wk = warp_codec_info(block, false, scheme.code);
        const int64_t want = (nblocks + wk.tile_blocks - 1) / wk.tile_blocks;
        const int64_t cap = static_cast<int64_t>(dev->sm_count) * 16;
        const cudaError_t e = launch_warp_decompress(block, scheme, packed_in, y_bf16_out, nblocks,
                                                     static_cast<int>(want < cap ? want : cap),
                                                     reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? TACO_OK : cuda_fail(e);
    }
    // Tensor-core kernel over tiles of 128 (B = 64: 256) blocks: one CTA per
    // tile, of which one per SM runs and takes the tiles of CTAs it cancels.
    const KernelInfo ki = decompress_kernel_info(block, scheme.code);
    const int64_t ntiles = (nblocks + ki.tile_blocks - 1) / ki.tile_blocks;
    if (ntiles > INT32_MAX)
        return TACO_ERR_BAD_SHAPE;
    alignas(64) CUtensorMap map;
    const int re = view_row_elems(block), rows_per_block = block / re;
    cudaError_t e = encode_block_rows_map(&map, y_bf16_out, nblocks * rows_per_block, re,
                                          ki.tile_blocks * rows_per_block);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const int grid = static_cast<int>(ntiles);
    e = launch_decompress(block, scheme, &map, packed_in, nblocks, dev->fault, grid,
                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TACO_OK : cuda_fail(e);
}

taco_status_t reduce_impl(const void *const *packed_shards, int num_shards, int64_t rows, int64_t hidden, int block,
                          Scheme scheme, void *packed_out, taco_stream_t stream)
{
    int64_t n = 0, bytes = 0;
    taco_status_t st = check_shape(rows, hidden, block, &n, &bytes);
    if (st != TACO_OK)
        return st;
    if (num_shards < 1 || num_shards > TACO_MAX_SHARDS)
        return TACO_ERR_BAD_SHARDS;
    if (n == 0)
        return TACO_OK;
    if (!packed_shards || !packed_out)
        return TACO_ERR_NULL_POINTER;
    ReduceArgs args{};
    for (int p = 0; p < num_shards; p++) {
        if (!packed_shards[p])
            return TACO_ERR_NULL_POINTER;
        if (!aligned16(packed_shards[p]))
            return TACO_ERR_MISALIGNED;
        if (overlap(packed_shards[p], bytes, packed_out, bytes))
            return TACO_ERR_OVERLAP;
        args.shards[p] = static_cast<const uint8_t *>(packed_shards[p]);
    }
    if (!aligned16(packed_out))
        return TACO_ERR_MISALIGNED;
    DeviceState *dev = nullptr;
    if ((st = device_state(&dev)) != TACO_OK)
        return st;
    args.out = static_cast<uint8_t *>(packed_out);
    args.nblocks = n / block;
    args.num_shards = num_shards;
    args.variant = scheme.variant;
    // One CTA per tile of blocks; one per SM runs and takes the tiles of CTAs
    // it cancels before they start.
    const KernelInfo ki = reduce_kernel_info(block, scheme.code, num_shards);
    const int64_t ntiles = (args.nblocks + ki.tile_blocks - 1) / ki.tile_blocks;
    if (ntiles > INT32_MAX)
        return TACO_ERR_BAD_SHAPE;
    const int grid = static_cast<int>(ntiles);
    const cudaError_t e =
        launch_reduce(block, scheme.code, args, dev->fault, grid, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TACO_OK : cuda_fail(e);
}

constexpr Scheme kMethod{TACO_VARIANT_ASH_DS, TACO_CODE_E4M3};

}  // namespace
cudaError_t launch_encode_selftest(int code, uint32_t first, int64_t count, void *codes, int grid,
                                   cudaStream_t stream);   // taco_selftest.cu

}  // namespace taco

using namespace taco;

extern "C" {

int64_t taco_compressed_bytes(int64_t rows, int64_t hidden, int block)
{
    int64_t n = 0, bytes = 0;
    if (check_shape(rows, hidden, block, &n, &bytes) != TACO_OK)
        return -1;
    return bytes;
}

taco_status_t taco_compress(const void *x_bf16, int64_t rows, int64_t hidden, int block, void *packed_out,
                            taco_stream_t stream)
{
    return compress_impl(x_bf16, rows, hidden, block, kMethod, packed_out, stream);
}

taco_status_t taco_decompress(const void *packed_in, int64_t rows, int64_t hidden, int block, void *y_bf16_out,
                              taco_stream_t stream)
{
    return decompress_impl(packed_in, rows, hidden, block, kMethod, y_bf16_out, stream);
}

taco_status_t taco_reduce_shards(const void *const *packed_shards, int num_shards, int64_t rows, int64_t hidden,
                                 int block, void *packed_out, taco_stream_t stream)
{
    return reduce_impl(packed_shards, num_shards, rows, hidden, block, kMethod, packed_out, stream);
}

taco_status_t taco_compress_ex(const void *x_bf16, int64_t rows, int64_t hidden, const taco_options_t *options,
                               void *packed_out, taco_stream_t stream)
{
    Scheme scheme{};
    const taco_status_t st = check_options(options, &scheme);
    if (st != TACO_OK)
        return st;
    return compress_impl(x_bf16, rows, hidden, options->block, scheme, packed_out, stream);
}

taco_status_t taco_decompress_ex(const void *packed_in, int64_t rows, int64_t hidden, const taco_options_t *options,
                                 void *y_bf16_out, taco_stream_t stream)
{
    Scheme scheme{};
    const taco_status_t st = check_options(options, &scheme);
    if (st != TACO_OK)
        return st;
    return decompress_impl(packed_in, rows, hidden, options->block, scheme, y_bf16_out, stream);
}

taco_status_t taco_reduce_shards_ex(const void *const *packed_shards, int num_shards, int64_t rows, int64_t hidden,
                                    const taco_options_t *options, void *packed_out, taco_stream_t stream)
{
    Scheme scheme{};
    const taco_status_t st = check_options(options, &scheme);
    if (st != TACO_OK)
        return st;
    return reduce_impl(packed_shards, num_shards, rows, hidden, options->block, scheme, packed_out, stream);
}

taco_status_t taco_selftest_encode_bits(int code, uint32_t first, int64_t count, void *codes_out,
                                        taco_stream_t stream)
{
    if (code < TACO_CODE_E4M3 || code > TACO_CODE_INT8)
        return TACO_ERR_BAD_OPTIONS;
    if (count < 0 || count % 4 != 0 || first % 4 != 0 || count > (int64_t{1} << 32))
        return TACO_ERR_BAD_SHAPE;
    if (count == 0)
        return TACO_OK;
    if (!codes_out)
        return TACO_ERR_NULL_POINTER;
    if (!aligned16(codes_out))
        return TACO_ERR_MISALIGNED;
    DeviceState *dev = nullptr;
    const taco_status_t st = device_state(&dev);
    if (st != TACO_OK)
        return st;
    const int64_t want = (count / 4 + 255) / 256, cap = static_cast<int64_t>(dev->sm_count) * 8;
    const cudaError_t e = launch_encode_selftest(code, first, count, codes_out, static_cast<int>(want < cap ? want : cap),
                                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TACO_OK : cuda_fail(e);
}

taco_status_t taco_selftest_wait_timeout(taco_stream_t stream)
{
    DeviceState *dev = nullptr;
    const taco_status_t st = device_state(&dev);
    if (st != TACO_OK)
        return st;
    const cudaError_t e = launch_wait_selftest(dev->fault, 2000000ull, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TACO_OK : cuda_fail(e);
}

taco_status_t taco_device_status(taco_stream_t stream, uint32_t *flags_out)
{
    DeviceState *dev = nullptr;
    taco_status_t st = device_state(&dev);
    if (st != TACO_OK)
        return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    uint32_t flags = 0;
    if (e == cudaSuccess)
        e = cudaMemcpy(&flags, dev->fault, sizeof flags, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && flags != 0) {
        const uint32_t zero = 0;
        e = cudaMemcpy(dev->fault, &zero, sizeof zero, cudaMemcpyHostToDevice);
    }
    if (flags_out)
        *flags_out = flags;
    if (e != cudaSuccess)
        return cuda_fail(e);
    return flags ? TACO_ERR_DEVICE_FAULT : TACO_OK;
}

const char *taco_status_string(taco_status_t status)
{
    switch (status) {
    case TACO_OK: return "TACO_OK";
    case TACO_ERR_NULL_POINTER: return "TACO_ERR_NULL_POINTER: a required pointer is NULL";
    case TACO_ERR_BAD_SHAPE: return "TACO_ERR_BAD_SHAPE: rows/hidden negative, hidden not a multiple of the block, or too large";
    case TACO_ERR_UNSUPPORTED_BLOCK: return "TACO_ERR_UNSUPPORTED_BLOCK: block must be 32, 64, 128, 256 or 512";
    case TACO_ERR_MISALIGNED: return "TACO_ERR_MISALIGNED: device pointers must be 16-byte aligned";
    case TACO_ERR_BAD_SHARDS: return "TACO_ERR_BAD_SHARDS: num_shards must be in [1, 16]";
    case TACO_ERR_OVERLAP: return "TACO_ERR_OVERLAP: an output overlaps an input";
    case TACO_ERR_CUDA: return "TACO_ERR_CUDA: a CUDA call failed (see taco_last_cuda_error)";
    case TACO_ERR_DEVICE_FAULT: return "TACO_ERR_DEVICE_FAULT: a kernel gave up waiting for a copy";
    case TACO_ERR_BAD_OPTIONS: return "TACO_ERR_BAD_OPTIONS: options NULL, or unknown variant or code format";
    default: return "unknown taco_status_t";
    }
}

int taco_last_cuda_error(void)
{
    return t_last_cuda_error;
}

int taco_abi_version(void)
{
    return TACO_ABI_VERSION;
}

}  // extern "C"
