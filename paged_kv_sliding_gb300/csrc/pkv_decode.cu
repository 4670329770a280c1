// Paged decode: host launch of the kernels in pkv_decode_kernel.cuh. This unit
// instantiates the bf16-cache kernels and dispatches the 8-bit ones to
// pkv_decode_fp8.cu (two units, so the build compiles them in parallel).
#include "pkv_decode_kernel.cuh"

namespace pkv {

bool encode_kv_map(CUtensorMap *m, const void *base, int head_dim, int num_kv_heads, int page_size,
                   int num_pages, int box_rows, int kv_dtype)
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    const int eb = kv_dtype == PKV_BF16 ? 2 : 1;
    if (eb == 2) {
        // bf16: the pool as 5-D [8-row blocks][H_kv][128-byte plane][row in block][64]
        // (a page of a multiple of 8 rows is a run of 8-row blocks); a box of box_rows
        // rows of one KV head and every plane lands as box_rows / 8 group-major row
        // groups of the kernel's stage.
        const cuuint64_t row = (cuuint64_t)num_kv_heads * head_dim * 2;
        const cuuint64_t blocks = (cuuint64_t)(num_pages > 0 ? num_pages : 1) * (cuuint64_t)page_size / 8;
        const cuuint64_t dims5[5] = {64, 8, (cuuint64_t)head_dim / 64, (cuuint64_t)num_kv_heads, blocks};
        const cuuint64_t strides5[4] = {row, 128, (cuuint64_t)head_dim * 2, 8 * row};
        const cuuint32_t box5[5] = {64, 8, (cuuint32_t)head_dim / 64, 1, (cuuint32_t)box_rows / 8};
        const cuuint32_t estr5[5] = {1, 1, 1, 1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims5, strides5, box5, estr5,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    // 8-bit: boxes of one 128-byte plane (128 elements) x rows of one page; an 8-bit row
    // of d 64 is a single 64-byte plane with the 64-byte swizzle.
    const int row_bytes = head_dim * eb;
    const int plane = row_bytes < 128 ? row_bytes : 128;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)page_size,
                                (cuuint64_t)(num_pages > 0 ? num_pages : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)row_bytes, (cuuint64_t)num_kv_heads * row_bytes,
                                   (cuuint64_t)page_size * num_kv_heads * row_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)(plane / eb), 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              plane == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_tma_page_size(int page_size, int tile)
{
    // whole pages inside a stage, or whole stages inside a page
    if (page_size < 8 || page_size % 8 != 0)
        return false;
    return page_size <= tile ? tile % page_size == 0 : page_size % tile == 0;
}

cudaError_t launch_decode(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s, int tile,
                          bool overlap_prev)
{
    using dec::launch_decode_dt;
    if (tile == 32 && head_dim > 128)
        return cudaErrorInvalidValue;
    const int tt = decode_kernel_tile(tile, head_dim, p.kv_dtype);
    const bool tma = decode_tma_page_size(p.page_size, tt);
    CUtensorMap tk{}, tv{};
    if (tma) {
        const int rows = p.page_size < tt ? p.page_size : tt;
        if (!encode_kv_map(&tk, p.k_cache, head_dim, p.num_kv_heads, p.page_size, p.num_pages, rows, p.kv_dtype) ||
            !encode_kv_map(&tv, p.v_cache, head_dim, p.num_kv_heads, p.page_size, p.num_pages, rows, p.kv_dtype))
            return cudaErrorInvalidValue;
    }
    if (p.kv_dtype != PKV_BF16)
        return launch_decode_kv8(p, head_dim, num_items, s, tile, tma, tk, tv, overlap_prev);
    constexpr int BF = PKV_BF16;
    if (tile == 32) {
        switch (head_dim) {
        case 64: return tma ? launch_decode_dt<64, true, 32, BF>(p, tk, tv, num_items, s, overlap_prev)
                            : launch_decode_dt<64, false, 32, BF>(p, tk, tv, num_items, s, overlap_prev);
        case 128: return tma ? launch_decode_dt<128, true, 32, BF>(p, tk, tv, num_items, s, overlap_prev)
                             : launch_decode_dt<128, false, 32, BF>(p, tk, tv, num_items, s, overlap_prev);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (head_dim) {
    case 64: return tma ? launch_decode_dt<64, true, 64, BF>(p, tk, tv, num_items, s, overlap_prev)
                        : launch_decode_dt<64, false, 64, BF>(p, tk, tv, num_items, s, overlap_prev);
    case 128: return tma ? launch_decode_dt<128, true, 64, BF>(p, tk, tv, num_items, s, overlap_prev)
                         : launch_decode_dt<128, false, 64, BF>(p, tk, tv, num_items, s, overlap_prev);
    case 256: return tma ? launch_decode_dt<256, true, 64, BF>(p, tk, tv, num_items, s, overlap_prev)
                         : launch_decode_dt<256, false, 64, BF>(p, tk, tv, num_items, s, overlap_prev);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
