// Paged prefill / extend over 8-bit K/V caches (E4M3 or E5M2, torch.float8_e4m3fn /
// torch.float8_e5m2 in flashinfer_backend.py): the kernels of pkv_prefill_kernel.cuh
// instantiated for one-byte elements. Q and the caches are read with plain and
// cp.async loads, so no tensor map is used.
#include "pkv_prefill_kernel.cuh"

namespace pkv {
namespace {

template <int KV>
cudaError_t launch_kv(const PrefillParams &p, int head_dim, int mask_mode, int num_ctas, cudaStream_t s)
{
    const CUtensorMap none{};
    switch (head_dim) {
    case 64: return pp::launch_pp_dt<64, false, false, KV>(p, mask_mode, none, none, none, none, num_ctas, s);
    case 128: return pp::launch_pp_dt<128, false, false, KV>(p, mask_mode, none, none, none, none, num_ctas, s);
    case 256: return pp::launch_pp_dt<256, false, false, KV>(p, mask_mode, none, none, none, none, num_ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prefill_pp_kv8(const PrefillParams &p, int head_dim, int mask_mode, int num_ctas,
                                  cudaStream_t s)
{
    if (p.ragged)
        return cudaErrorInvalidValue;
    if (p.kv_dtype == PKV_FP8_E4M3)
        return launch_kv<PKV_FP8_E4M3>(p, head_dim, mask_mode, num_ctas, s);
    if (p.kv_dtype == PKV_FP8_E5M2)
        return launch_kv<PKV_FP8_E5M2>(p, head_dim, mask_mode, num_ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
