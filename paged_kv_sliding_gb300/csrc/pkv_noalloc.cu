// Decode through a single call that allocates no device memory.
//
// pkv_plan_create / pkv_run keep their work list and split-KV partial states in a
// workspace the plan obtains with cudaMalloc. Some callers cannot do that: serving
// processes whose memory pool has already reserved the device memory and that
// forbid further driver allocations, and latency-critical paths that cannot pay
// for cudaMalloc / cudaFree, which may synchronise the whole device.
// pkv_decode_noalloc serves them: the work list and the partial states live in one
// file-scope __device__ array of kScratchBytes, which every GPU that loads this
// library holds until the process exits.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "pkv_internal.h"
#include "pkv_nvtx.h"

namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

int noalloc_fail(int status, const std::string &msg)
{
    pkv::set_last_error(("pkv_decode_noalloc: " + msg).c_str());
    return status;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of g_scratch on the current device, looked up once per device
// (cudaGetSymbolAddress with that device current; the host-side symbol itself is
// only a stand-in and must never reach a kernel).
int scratch_address(void **out)
{
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return noalloc_fail(PKV_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(PKV_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        ce = cudaGetSymbolAddress(&p, g_scratch);
        if (ce != cudaSuccess || !p)
            return noalloc_fail(PKV_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(ce));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

// The work list reaches the device as the by-value arguments of small copy kernels
// (a kernel's argument block may hold up to 32764 bytes): no host staging buffer
// has to outlive the call, and nothing makes the host wait for earlier work on the
// stream, as a copy from pageable host memory would.
constexpr int kUploadWords = 2040;  // 16-byte words per copy kernel (32640 bytes)

struct UploadBlock {
    uint4 *dst;
    int32_t words;
    int32_t pad;
    uint4 data[kUploadWords];
};
static_assert(sizeof(UploadBlock) <= 32764, "kernel argument block");

__global__ void __launch_bounds__(256) upload_kernel(const __grid_constant__ UploadBlock blk)
{
    for (int i = threadIdx.x; i < blk.words; i += blockDim.x)
        blk.dst[i] = blk.data[i];
}

// Copy `bytes` (a multiple of 16) from host memory to device address `dst`, one copy
// kernel per kUploadWords words, enqueued on `stream`.
cudaError_t upload(uint8_t *dst, const uint8_t *src, size_t bytes, cudaStream_t stream)
{
    static thread_local UploadBlock blk;  // argument staging; launches copy it out
    const size_t words = bytes / 16;
    for (size_t w0 = 0; w0 < words; w0 += kUploadWords) {
        const size_t n = std::min<size_t>(kUploadWords, words - w0);
        blk.dst = reinterpret_cast<uint4 *>(dst) + w0;
        blk.words = (int32_t)n;
        blk.pad = 0;
        std::memcpy(blk.data, src + 16 * w0, 16 * n);
        upload_kernel<<<1, 256, 0, stream>>>(blk);
        const cudaError_t ce = cudaGetLastError();
        if (ce != cudaSuccess)
            return ce;
    }
    return cudaSuccess;
}

int page_shift(int page_size)
{
    if (page_size <= 0 || (page_size & (page_size - 1)))
        return -1;
    int s = 0;
    while ((1 << s) < page_size)
        ++s;
    return s;
}

}  // namespace

extern "C" int pkv_decode_noalloc(const pkv_plan_desc *d, const void *q, const void *k_cache,
                                  const void *v_cache, void *out, float *lse, void *stream_)
{
    using namespace pkv;
    NvtxRange range("pkv_decode_noalloc");
    pkv::set_last_error("");
    if (!d || d->kind != PKV_DECODE)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "needs a PKV_DECODE description");
    const int B = d->batch_size;
    if (B < 0 || !d->kv_indptr || !d->kv_last_page_len)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "batch_size, kv_indptr and kv_last_page_len are required");
    if (d->num_qo_heads <= 0 || d->num_kv_heads <= 0 || d->num_qo_heads % d->num_kv_heads)
        return noalloc_fail(PKV_ERR_UNSUPPORTED, "head counts");
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return noalloc_fail(PKV_ERR_UNSUPPORTED, "head_dim not in {64, 128, 256}");
    if (d->page_size <= 0 || d->num_pages < 0 || d->dtype != PKV_BF16)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "page_size, num_pages or dtype");
    if (d->kv_dtype != PKV_BF16)
        return noalloc_fail(PKV_ERR_UNSUPPORTED, "bf16 caches only (kv_dtype must be PKV_BF16)");
    for (float x : {d->logits_soft_cap, d->k_scale, d->v_scale})
        if (!(x == x) || std::isinf(x))
            return noalloc_fail(PKV_ERR_INVALID_ARG, "logits_soft_cap, k_scale and v_scale must be finite");
    if (!(d->sm_scale > 0.f) || std::isinf(d->sm_scale))
        return noalloc_fail(PKV_ERR_UNSUPPORTED, "sm_scale must be positive and finite");
    if (d->kv_indptr[0] != 0)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "kv_indptr[0] must be 0");
    if (B > 0 && d->kv_indptr[B] > 0 && !d->kv_indices)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "kv_indices is NULL");
    if (B > 0 && (!q || !out || !k_cache || !v_cache))
        return noalloc_fail(PKV_ERR_INVALID_ARG, "q, caches and out are required");
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out) % 16 || (uintptr_t)lse % 4)
        return noalloc_fail(PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned, lse 4-byte");
    if (B == 0)
        return PKV_OK;

    const int group = d->num_qo_heads / d->num_kv_heads;
    const int W = d->window_left < 0 ? -1 : d->window_left;
    const bool causal = d->causal != 0;
    const int head_blocks = (group + kDecodeRows - 1) / kDecodeRows;

    // Requests and their visible key intervals (one query row each).
    std::vector<RequestInfo> reqs(B);
    std::vector<int64_t> lo(B), len(B);
    for (int b = 0; b < B; ++b) {
        const int64_t np = (int64_t)d->kv_indptr[b + 1] - d->kv_indptr[b];
        if (np < 0)
            return noalloc_fail(PKV_ERR_INVALID_ARG, "kv_indptr decreases");
        const int64_t last = d->kv_last_page_len[b];
        if (np > 0 && (last < 1 || last > d->page_size))
            return noalloc_fail(PKV_ERR_INVALID_ARG, "kv_last_page_len outside [1, page_size]");
        const int64_t kv_len = np > 0 ? (np - 1) * d->page_size + last : 0;
        const int64_t p = d->q_start ? (int64_t)d->q_start[b] : kv_len - 1;
        if (kv_len > INT32_MAX / 2 || std::llabs(p) > INT32_MAX / 2)
            return noalloc_fail(PKV_ERR_UNSUPPORTED, "request too long");
        reqs[b] = {b, 1, (int32_t)kv_len, (int32_t)d->kv_indptr[b], (int32_t)p, 0, 0, 0};
        lo[b] = W >= 0 ? std::max<int64_t>(0, p - W) : 0;
        const int64_t hi = causal ? std::min<int64_t>(kv_len - 1, p) : kv_len - 1;
        len[b] = std::max<int64_t>(0, hi - lo[b] + 1);
    }
    // Split size: the caller's, none, or 1024 keys when the batch alone cannot
    // fill two CTAs per SM.
    int64_t chunk = INT32_MAX;
    if (!d->disable_split_kv) {
        if (d->fixed_split_size > 0) {
            chunk = d->fixed_split_size;
        } else {
            int dev = 0, sms = 148;
            if (cudaGetDevice(&dev) == cudaSuccess)
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if ((int64_t)B * d->num_kv_heads * head_blocks < 2LL * sms)
                chunk = 1024;
        }
    }
    std::vector<DecodeItem> items;
    std::vector<MergeItem> merges;
    int32_t num_partials = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t n = len[b] > 0 ? (len[b] + chunk - 1) / chunk : 1;
        int32_t pbase = -1;
        if (n > 1) {
            pbase = num_partials;
            num_partials += (int32_t)n;
            merges.push_back({b, pbase, (int32_t)n, 0});
        }
        for (int64_t s = 0; s < n; ++s) {
            const int64_t j0 = lo[b] + s * chunk;
            const int64_t j1 = len[b] > 0 ? std::min(lo[b] + len[b], j0 + chunk) : j0;
            for (int hk = 0; hk < d->num_kv_heads; ++hk)
                for (int h0 = 0; h0 < group; h0 += kDecodeRows)
                    items.push_back({b, hk, hk * group + h0, std::min(kDecodeRows, group - h0), (int32_t)j0,
                                     (int32_t)j1, n > 1 ? (int32_t)(pbase + s) : -1, pbase, (int32_t)n, -1,
                                     reqs[b].qo_begin, reqs[b].kv_len, reqs[b].kv_page_begin, 0});
        }
    }
    std::stable_sort(items.begin(), items.end(),
                     [](const DecodeItem &a, const DecodeItem &c) { return (a.j1 - a.j0) > (c.j1 - c.j0); });

    // Scratch layout: status | requests | items | merge items | partial lse | partial o.
    size_t off = 0;
    const size_t o_status = off;
    off = align_up(off + sizeof(int32_t), 256);
    const size_t o_reqs = off;
    off = align_up(off + sizeof(RequestInfo) * reqs.size(), 256);
    const size_t o_items = off;
    off = align_up(off + sizeof(DecodeItem) * items.size(), 256);
    const size_t o_merge = off;
    off = align_up(off + sizeof(MergeItem) * std::max<size_t>(1, merges.size()), 256);
    const size_t o_pl = off;
    off = align_up(off + sizeof(float) * (size_t)num_partials * d->num_qo_heads, 256);
    const size_t o_po = off;
    off = align_up(off + sizeof(float) * (size_t)num_partials * d->num_qo_heads * d->head_dim, 256);
    if (off > kScratchBytes)
        return noalloc_fail(PKV_ERR_UNSUPPORTED,
                            "the batch needs " + std::to_string(off) + " bytes of scratch, above the " +
                                std::to_string(kScratchBytes) + "-byte limit (use fewer splits or pkv_run)");

    void *base_v = nullptr;
    int st = scratch_address(&base_v);
    if (st != PKV_OK)
        return st;
    uint8_t *base = (uint8_t *)base_v;
    cudaStream_t stream = (cudaStream_t)stream_;

    // One host image of everything before the partial states, carried to the device
    // in the arguments of the copy kernels (their launches copy it out, so the image
    // may be freed on return).
    std::vector<uint8_t> image(o_pl, 0);
    std::memcpy(image.data() + o_reqs, reqs.data(), sizeof(RequestInfo) * reqs.size());
    std::memcpy(image.data() + o_items, items.data(), sizeof(DecodeItem) * items.size());
    if (!merges.empty())
        std::memcpy(image.data() + o_merge, merges.data(), sizeof(MergeItem) * merges.size());
    cudaError_t ce = upload(base, image.data(), image.size(), stream);
    if (ce != cudaSuccess)
        return noalloc_fail(PKV_ERR_CUDA, std::string("uploading the work list: ") + cudaGetErrorString(ce));
    // The array keeps the previous call's contents: the status word must restart
    // at zero (the staging image above already holds a zero there; the partial
    // states need no clearing, every slot is written before it is read).

    DecodeParams p{};
    p.items = (const DecodeItem *)(base + o_items);
    p.reqs = (const RequestInfo *)(base + o_reqs);
    p.kv_indices = d->kv_indices;
    p.q = (const uint16_t *)q;
    p.k_cache = (const uint16_t *)k_cache;
    p.v_cache = (const uint16_t *)v_cache;
    p.out = (uint16_t *)out;
    p.lse = lse;
    p.partial_o = (float *)(base + o_po);
    p.partial_lse = (float *)(base + o_pl);
    p.status = (int32_t *)(base + o_status);
    p.num_qo_heads = d->num_qo_heads;
    p.num_kv_heads = d->num_kv_heads;
    p.page_size = d->page_size;
    p.page_shift = page_shift(d->page_size);
    p.num_pages = d->num_pages;
    const LogitFactors lf = logit_factors(*d);
    p.sm_scale_log2 = lf.sm_scale_log2;
    p.cap_in = lf.cap_in;
    p.cap_out = lf.cap_out;
    p.v_scale = lf.v_scale;
    p.wait_ns = wait_ns_of(*d);  // no status to report a probe's expiry: never probed
    int64_t max_keys = 0;
    for (const DecodeItem &it : items)
        max_keys = std::max<int64_t>(max_keys, it.j1 - it.j0);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // No overlap with the copy kernels: the decode reads its work item first thing.
    ce = launch_decode(p, d->head_dim, (int)items.size(), stream,
                       decode_tile_for(d->head_dim, max_keys, (int64_t)items.size(), sms), false);
    if (ce != cudaSuccess)
        return noalloc_fail(PKV_ERR_CUDA, std::string("decode launch: ") + cudaGetErrorString(ce));
    if (!merges.empty()) {
        MergePartialsParams m{};
        m.items = (const MergeItem *)(base + o_merge);
        m.partial_o = p.partial_o;
        m.partial_lse = p.partial_lse;
        m.out = (uint16_t *)out;
        m.lse = lse;
        m.num_items = (int32_t)merges.size();
        m.num_qo_heads = d->num_qo_heads;
        m.v_scale = p.v_scale;
        ce = launch_merge_partials(m, d->head_dim, stream);
        if (ce != cudaSuccess)
            return noalloc_fail(PKV_ERR_CUDA, std::string("merge launch: ") + cudaGetErrorString(ce));
    }
    return PKV_OK;
}
