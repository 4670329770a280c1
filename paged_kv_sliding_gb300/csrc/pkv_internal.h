// Internal declarations shared by the host plan code and the kernels of libpkv.
// Not part of the C ABI (include/pkv.h is).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

// Per-request facts the kernels need, computed once by the plan.
struct RequestInfo {
    int32_t qo_begin;       // first global query row (qo_indptr[b])
    int32_t qo_len;         // query rows of the request
    int32_t kv_len;         // valid tokens in its pages
    int32_t kv_page_begin;  // kv_indptr[b]
    int32_t q_start;        // position of its first query row
    int32_t pad0, pad1, pad2;
};

// One work item of the prefill kernel: one or two tiles of packed query rows (query
// tokens x the KV head's query-head group) of one request against the kv_tiles KV
// tiles from key kv_start on, which cover every key its positions can see.
struct PrefillItem {
    int32_t req;
    int32_t kv_head;
    int32_t tok0;        // first query token of the tile, within the request
    int32_t ntok;        // query tokens in the tile
    int32_t kv_start;    // first key of the item's first KV tile (aligned for the loader)
    int32_t kv_tiles;    // KV tiles of the item (0: no visible key)
    int32_t kv_tile_rot; // tiles are visited from tile kv_tile_rot on, wrapping around
    int32_t pad0;
};

// First key of the KV tile visited at step j (0 <= j < kv_tiles) of a prefill item
// whose tiles hold T keys. Softmax accumulation is order-independent; staggering the
// start keeps the items that run at the same time on one KV head from all missing L2
// on the same tile.
__host__ __device__ inline int prefill_kv_key_at(const PrefillItem &it, int j, int T)
{
    const int k = j + it.kv_tile_rot;
    return it.kv_start + (k < it.kv_tiles ? k : k - it.kv_tiles) * T;
}

// One CTA of the decode kernel: up to kDecodeRows query heads of one request's
// single row against the key range [j0, j1) of one KV head.
struct DecodeItem {
    int32_t req;
    int32_t kv_head;
    int32_t head0;    // first query head handled
    int32_t nheads;   // query heads handled (<= kDecodeRows)
    int32_t j0, j1;   // key range, already clipped to the visible interval
    int32_t partial;  // -1: write out/lse directly; else partial slot of this split
    int32_t pbase;    // first partial slot of the request (split items)
    int32_t nsplit;   // splits of the request (split items)
    int32_t counter;  // arrival counter of this (request, KV head, head block) group
    // The request's facts the kernel needs, carried here so that a CTA's first
    // page-table read does not wait behind a second dependent load.
    int32_t row;            // the request's query row (its qo_begin)
    int32_t kv_len;         // keys in the request's cache
    int32_t kv_page_begin;  // the request's first entry in kv_indices
    int32_t pad0;
};

// Merge of a request's split-KV partial states into its output row.
struct MergeItem {
    int32_t row;            // global query row
    int32_t partial_begin;  // first partial slot
    int32_t num_partials;   // splits to combine
    int32_t pad;
};

constexpr int kDecodeRows = 16;   // query heads per decode CTA (one m16 MMA tile)
constexpr int kPrefillRows = 128; // packed query rows per prefill CTA (UMMA M)

enum MaskMode : int32_t { kMaskNone = 0, kMaskCausal = 1, kMaskCausalWindow = 2, kMaskWindow = 3 };

struct DecodeParams {
    const DecodeItem *items;
    const int32_t *live_items;  // non-NULL: CTAs at or above *live_items have no work
    const RequestInfo *reqs;
    const int32_t *kv_indices;
    const uint16_t *q;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    uint16_t *out;
    float *lse;          // may be null
    float *partial_o;    // [num_partials, num_qo_heads, head_dim]
    float *partial_lse;  // [num_partials, num_qo_heads]
    int32_t *merge_counters;  // non-null: the last split CTA of a group merges its partials
    int32_t *status;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t page_size;
    int32_t page_shift;  // log2(page_size) when a power of two, else -1
    int32_t num_pages;
    float sm_scale_log2; // sm_scale * k_scale * log2(e)
    float cap_in;        // soft cap: dot -> cap_out * tanh(dot * cap_in); cap_in = 0: none
    float cap_out;
    float v_scale;       // multiplies the final output
    int32_t kv_dtype;    // element type of the caches (pkv_dtype: bf16 or an 8-bit float)
    int32_t wait_probe;  // nonzero: each CTA's first consuming wait is on a barrier nothing completes
    long long wait_ns;   // bound of every wait (globaltimer nanoseconds)
};

struct MergePartialsParams {
    const MergeItem *items;
    const float *partial_o;
    const float *partial_lse;
    uint16_t *out;
    float *lse;
    int32_t num_items;
    int32_t num_qo_heads;
    float v_scale;  // multiplies the merged output
};

struct PrefillParams {
    const PrefillItem *items;    // grouped by CTA
    const int32_t *cta_items;    // CTA c runs items [cta_items[c], cta_items[c + 1])
    const RequestInfo *reqs;
    const int32_t *kv_indices;
    const uint16_t *q;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    uint16_t *out;
    float *lse;
    int32_t *status;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;           // num_qo_heads / num_kv_heads
    int32_t tokens_per_tile; // query tokens per CTA = floor(128 / group)
    int32_t page_size;
    int32_t page_shift;
    int32_t num_pages;
    int32_t window_left;
    int32_t total_q;         // rows of q (bound of the query tensor map)
    float sm_scale_log2;     // sm_scale * k_scale * log2(e)
    float cap_in;            // soft cap, as in DecodeParams
    float cap_out;
    float v_scale;
    int32_t ragged;          // 1: K/V are contiguous [total_kv, H_kv, d], kv_page_begin = token offset
    int32_t total_kv;        // ragged: rows of K/V (bound of their tensor maps)
    int32_t kv_dtype;        // element type of the caches (pkv_dtype: bf16 or an 8-bit float)
    int32_t wait_probe;      // as in DecodeParams
    long long wait_ns;       // as in DecodeParams
};

// Bound of every wait inside the kernels: the descriptor's wait_limit_us, or 2 s.
constexpr long long kDefaultWaitNs = 2000000000LL;
inline long long wait_ns_of(const pkv_plan_desc &d)
{
    return d.wait_limit_us > 0 ? (long long)d.wait_limit_us * 1000LL : kDefaultWaitNs;
}

// The logit and output factors of a plan descriptor (k_scale folded into the logit
// scale; scales <= 0 mean 1; a soft cap <= 0 means none).
struct LogitFactors {
    float sm_scale_log2, cap_in, cap_out, v_scale;
};
inline LogitFactors logit_factors(const pkv_plan_desc &d)
{
    const float ks = d.k_scale > 0.f ? d.k_scale : 1.f;
    const float vs = d.v_scale > 0.f ? d.v_scale : 1.f;
    const float s = d.sm_scale * ks;
    LogitFactors f;
    f.sm_scale_log2 = s * 1.4426950408889634f;
    f.cap_in = d.logits_soft_cap > 0.f ? s / d.logits_soft_cap : 0.f;
    f.cap_out = d.logits_soft_cap > 0.f ? d.logits_soft_cap / s : 0.f;
    f.v_scale = vs;
    return f;
}

// Launchers (one per kernel family); return cudaGetLastError() of the launch.
// tile: KV tokens per stage, 64 or (head_dim <= 128) 32. overlap_prev: the kernel's
// set-up may overlap the previous kernel in the stream (programmatic dependent
// launch); false when that kernel writes the work list the decode reads first.
cudaError_t launch_decode(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s, int tile,
                          bool overlap_prev = true);
// KV tile of the decode kernel (head_dim <= 128): 32 tokens (4 CTAs per SM) for
// short key ranges, which are latency-bound, and for medium ones (<= 1024 keys)
// whose CTAs need more than one wave at 2 per SM but fit in one at 4; otherwise 64
// (twice the bytes in flight per CTA, which long ranges need).
inline int decode_tile_for(int head_dim, int64_t max_keys, int64_t n_items, int n_sm)
{
    if (head_dim > 128)
        return 64;
    if (max_keys <= 192)
        return 32;
    if (max_keys <= 1024 && n_items > 2LL * n_sm && n_items <= 4LL * n_sm)
        return 32;
    return 64;
}
// KV tokens per stage of the decode kernel that runs a plan's tile variant (32: short
// key ranges; 64: the rest): 8-bit caches at head_dim <= 128 run both variants with
// two 16-token sub-blocks per compute warp, so their stages are twice as long (64 and
// 128 tokens).
inline int decode_kernel_tile(int tile, int head_dim, int kv_dtype)
{
    return (kv_dtype != PKV_BF16 && head_dim <= 128) ? 2 * tile : tile;
}
// Page sizes whose pages the decode kernel loads with TMA boxes of a `tile`-token stage.
bool decode_tma_page_size(int page_size, int tile);
// Tensor map over a cache of kv_dtype elements for the decode kernel's TMA page boxes:
// bf16, 5-D [8-row blocks][KV head][128-byte plane][row in block][64], one box = box_rows
// rows of one KV head with every plane (the group-major stage layout); 8-bit, 4-D
// [page, slot, KV head, d], one box = one 128-byte plane (64 bytes at d 64) x box_rows.
bool encode_kv_map(CUtensorMap *m, const void *base, int head_dim, int num_kv_heads, int page_size,
                   int num_pages, int box_rows, int kv_dtype);
// The 8-bit-cache decode kernels (p.kv_dtype = PKV_FP8_E4M3 or PKV_FP8_E5M2).
cudaError_t launch_decode_kv8(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s, int tile,
                              bool tma, const CUtensorMap &tk, const CUtensorMap &tv, bool overlap_prev);
cudaError_t launch_merge_partials(const MergePartialsParams &p, int head_dim, cudaStream_t s);
cudaError_t launch_merge_state(const void *v_a, const float *s_a, const void *v_b,
                               const float *s_b, void *v_out, float *s_out, int64_t rows,
                               int head_dim, int dtype, cudaStream_t s);
// One persistent CTA per entry of cta_items (num_ctas + 1 offsets).
cudaError_t launch_prefill_pp(const PrefillParams &p, int head_dim, int mask_mode, int num_ctas,
                              cudaStream_t s);
// Page sizes whose pages the prefill kernel loads with TMA boxes.
bool prefill_pp_tma_page_size(int page_size, int head_dim);
// The prefill kernels over 8-bit caches (p.kv_dtype = PKV_FP8_E4M3 or PKV_FP8_E5M2).
cudaError_t launch_prefill_pp_kv8(const PrefillParams &p, int head_dim, int mask_mode, int num_ctas,
                                  cudaStream_t s);

// Set the calling thread's pkv_last_error() text.
void set_last_error(const char *msg);

// KV tile (tokens) of the prefill kernels for a head_dim.
int prefill_kv_tile(int head_dim);
// Query tokens per prefill CTA: one 128-row tile (head_dim 256) or two (64, 128).
inline int prefill_tokens_per_cta(int head_dim, int group)
{
    const int tq = group < kPrefillRows ? kPrefillRows / group : 1;
    return head_dim <= 128 ? 2 * tq : tq;
}

}  // namespace pkv
