// Paged prefill / extend: host launch of the kernels in pkv_prefill_kernel.cuh (bf16
// caches; the 8-bit-cache kernels are instantiated in pkv_prefill_fp8.cu).
#include "pkv_prefill_kernel.cuh"

namespace pkv {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

bool encode_nd(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims, const cuuint64_t *strides,
               const cuuint32_t *box)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_4d(CUtensorMap *m, const void *base, const cuuint64_t dims[4], const cuuint64_t strides[3],
               const cuuint32_t box[4])
{
    return encode_nd(m, 4, base, dims, strides, box);
}

}  // namespace

bool prefill_pp_tma_page_size(int page_size, int head_dim)
{
    const int T = prefill_kv_tile(head_dim);
    if (page_size < 8 || page_size % 8 != 0)
        return false;
    return page_size <= T ? T % page_size == 0 : page_size % T == 0;
}

int prefill_kv_tile(int head_dim) { return head_dim >= 256 ? 64 : 128; }

cudaError_t launch_prefill_pp(const PrefillParams &p, int head_dim, int mask_mode, int num_ctas, cudaStream_t s)
{
    if (p.kv_dtype != PKV_BF16)
        return launch_prefill_pp_kv8(p, head_dim, mask_mode, num_ctas, s);
    const int g = p.group, tq = p.tokens_per_tile, Hkv = p.num_kv_heads, P = p.page_size;
    const bool tma_kv = p.ragged || prefill_pp_tma_page_size(P, head_dim);
    const int T = prefill_kv_tile(head_dim);
    CUtensorMap tm_q{}, tm_k{}, tm_v{}, tm_o{};
    {
        const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)g, (cuuint64_t)Hkv,
                                    (cuuint64_t)(p.total_q > 0 ? p.total_q : 1)};
        const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)g * head_dim * 2,
                                       (cuuint64_t)Hkv * g * head_dim * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)g, 1, (cuuint32_t)tq};
        if (!encode_4d(&tm_q, p.q, dims, strides, box))
            return cudaErrorInvalidValue;
        // the output, in the same shape (the one-query-tile kernels store full items' rows with it)
        if (!encode_4d(&tm_o, p.out, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    if (p.ragged) {
        // [total_kv][H_kv][d] viewed as 4-D with a unit outer dimension; box (64, 1, T, 1)
        const cuuint64_t rows = (cuuint64_t)(p.total_kv > 0 ? p.total_kv : 1);
        const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)Hkv, rows, 1};
        const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)Hkv * head_dim * 2,
                                       rows * Hkv * head_dim * 2};
        const cuuint32_t box[4] = {64, 1, (cuuint32_t)T, 1};
        if (!encode_4d(&tm_k, p.k_cache, dims, strides, box) || !encode_4d(&tm_v, p.v_cache, dims, strides, box))
            return cudaErrorInvalidValue;
        switch (head_dim) {
        case 64: return pp::launch_pp_dt<64, true, true, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
        case 128: return pp::launch_pp_dt<128, true, true, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
        case 256: return pp::launch_pp_dt<256, true, true, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
        default: return cudaErrorInvalidValue;
        }
    }
    if (tma_kv) {
        // The page pool as 5-D [8-row blocks][H_kv][column chunk][row in block][64 columns]
        // (rows within a page are H_kv * d apart, so pages of a multiple of 8 rows are
        // runs of 8-row blocks): a box of rows_box rows of one KV head and every chunk
        // lands as rows_box / 8 group-major key groups of the kernel's ring slot.
        const int rows_box = P < T ? P : T;
        const cuuint64_t row = (cuuint64_t)Hkv * head_dim * 2;
        const cuuint64_t blocks = (cuuint64_t)(p.num_pages > 0 ? p.num_pages : 1) * (cuuint64_t)P / 8;
        const cuuint64_t dims[5] = {64, 8, (cuuint64_t)head_dim / 64, (cuuint64_t)Hkv, blocks};
        const cuuint64_t strides[4] = {row, 128, (cuuint64_t)head_dim * 2, 8 * row};
        const cuuint32_t box[5] = {64, 8, (cuuint32_t)head_dim / 64, 1, (cuuint32_t)rows_box / 8};
        if (!encode_nd(&tm_k, 5, p.k_cache, dims, strides, box) || !encode_nd(&tm_v, 5, p.v_cache, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    switch (head_dim) {
    case 64:
        return tma_kv ? pp::launch_pp_dt<64, true, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s)
                      : pp::launch_pp_dt<64, false, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
    case 128:
        return tma_kv ? pp::launch_pp_dt<128, true, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s)
                      : pp::launch_pp_dt<128, false, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
    case 256:
        return tma_kv ? pp::launch_pp_dt<256, true, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s)
                      : pp::launch_pp_dt<256, false, false, PKV_BF16>(p, mask_mode, tm_q, tm_k, tm_v, tm_o, num_ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
