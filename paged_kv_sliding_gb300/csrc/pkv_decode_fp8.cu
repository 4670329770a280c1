// Paged decode over 8-bit K/V caches (E4M3 or E5M2, torch.float8_e4m3fn /
// torch.float8_e5m2 in flashinfer_backend.py should_use_tensor_core): the kernels of
// pkv_decode_kernel.cuh instantiated for one-byte elements. K and V tiles are
// widened to f16 in registers right before their MMAs; k_scale and v_scale
// dequantise through the logit scale and the output factor.
#include "pkv_decode_kernel.cuh"

namespace pkv {
namespace {

template <int KV>
cudaError_t launch_kv(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s, int tile, bool tma,
                      const CUtensorMap &tk, const CUtensorMap &tv, bool overlap_prev)
{
    using dec::launch_decode_dt;
    if (tile == 32) {
        // the short variant: 64-token stages, two compute warps of two 16-token
        // sub-blocks each, 4 CTAs per SM (decode_kernel_tile)
        switch (head_dim) {
        case 64: return tma ? launch_decode_dt<64, true, 64, KV, 32>(p, tk, tv, num_items, s, overlap_prev)
                            : launch_decode_dt<64, false, 64, KV, 32>(p, tk, tv, num_items, s, overlap_prev);
        case 128: return tma ? launch_decode_dt<128, true, 64, KV, 32>(p, tk, tv, num_items, s, overlap_prev)
                             : launch_decode_dt<128, false, 64, KV, 32>(p, tk, tv, num_items, s, overlap_prev);
        default: return cudaErrorInvalidValue;
        }
    }
    // the long variant: 128-token stages, two 16-token sub-blocks per compute warp
    // (decode_kernel_tile), except at head_dim 256
    switch (head_dim) {
    case 64: return tma ? launch_decode_dt<64, true, 128, KV, 32>(p, tk, tv, num_items, s, overlap_prev)
                        : launch_decode_dt<64, false, 128, KV, 32>(p, tk, tv, num_items, s, overlap_prev);
    case 128: return tma ? launch_decode_dt<128, true, 128, KV, 32>(p, tk, tv, num_items, s, overlap_prev)
                         : launch_decode_dt<128, false, 128, KV, 32>(p, tk, tv, num_items, s, overlap_prev);
    case 256: return tma ? launch_decode_dt<256, true, 64, KV>(p, tk, tv, num_items, s, overlap_prev)
                         : launch_decode_dt<256, false, 64, KV>(p, tk, tv, num_items, s, overlap_prev);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_decode_kv8(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s, int tile,
                              bool tma, const CUtensorMap &tk, const CUtensorMap &tv, bool overlap_prev)
{
    if (p.kv_dtype == PKV_FP8_E4M3)
        return launch_kv<PKV_FP8_E4M3>(p, head_dim, num_items, s, tile, tma, tk, tv, overlap_prev);
    if (p.kv_dtype == PKV_FP8_E5M2)
        return launch_kv<PKV_FP8_E5M2>(p, head_dim, num_items, s, tile, tma, tk, tv, overlap_prev);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
