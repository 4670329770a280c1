// Host side of libpkv: argument validation, the plan (work decomposition with the
// window fixed at plan time), run dispatch and error reporting.
//
// The plan follows the shape of the pages' plan/run split (sglang
// flashinfer_backend.py page: in section fast_prefill_plan the schedule comes from
// host-known query and KV layouts without a device-to-host read; in section
// call_begin_forward the plan receives kv_indptr, kv_indices and kv_last_page_len)
// with the change sglang PR #31501 asks for: window_left and causal are given to the
// plan, and the run cannot override them.
#include <algorithm>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include "pkv_internal.h"
#include "pkv_nvtx.h"

using namespace pkv;

namespace {

thread_local std::string g_last_error;

int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(e == cudaErrorMemoryAllocation ? PKV_ERR_OOM : PKV_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

void pkv::set_last_error(const char *msg) { g_last_error = msg ? msg : ""; }

struct pkv_plan {
    pkv_plan_desc desc{};  // host pointers cleared after planning
    int device = 0;
    int mask_mode = kMaskNone;
    int num_items = 0;
    int num_partials = 0;
    int num_ctas = 0;  // prefill: persistent CTAs (lists)
    int n_sm = 0;
    // Capturable plans: launch shapes and workspace sized by the declared capacity,
    // re-planned in place by pkv_plan_update through two pinned staging images.
    bool capturable = false;
    int64_t cap_items = 0, cap_total_q = 0, cap_batch = 0;
    size_t upload_bytes = 0;
    void *staging[2] = {nullptr, nullptr};
    cudaEvent_t staging_done[2] = {nullptr, nullptr};
    int staging_next = 0;
    int32_t *d_live = nullptr;  // live work items (capturable decode launches exit above it)
    int64_t total_kv = 0;       // ragged prefill: rows of the contiguous K/V
    int decode_tile = 64;  // decode: KV tokens per stage of the kernel
    int64_t total_q = 0;
    const int32_t *kv_indices = nullptr;  // borrowed device pointer
    void *workspace = nullptr;
    size_t workspace_bytes = 0;
    RequestInfo *d_reqs = nullptr;
    void *d_items = nullptr;
    int32_t *d_cta_items = nullptr;
    float *d_partial_o = nullptr;
    float *d_partial_lse = nullptr;
    int32_t *d_status = nullptr;
    int32_t *d_counters = nullptr;  // split-KV arrival counters (fused merge)
    cudaEvent_t ev_begin = nullptr;  // optional timing events around the main kernel
    cudaEvent_t ev_end = nullptr;
};

namespace {

struct HostRequest {
    int64_t qo_begin, qo_len, kv_len, kv_page_begin, q_start;
};

int validate(const pkv_plan_desc *d, std::vector<HostRequest> &reqs)
{
    if (!d)
        return fail(PKV_ERR_INVALID_ARG, "desc is NULL");
    if (d->kind != PKV_PREFILL && d->kind != PKV_DECODE && d->kind != PKV_PREFILL_RAGGED)
        return fail(PKV_ERR_INVALID_ARG, "kind %d is not a pkv_kind", d->kind);
    const bool ragged = d->kind == PKV_PREFILL_RAGGED;
    if (d->batch_size < 0)
        return fail(PKV_ERR_INVALID_ARG, "batch_size %d < 0", d->batch_size);
    const int B = d->batch_size;
    if (!d->kv_indptr || (!ragged && !d->kv_last_page_len))
        return fail(PKV_ERR_INVALID_ARG, "kv_indptr%s required", ragged ? " is" : " and kv_last_page_len are");
    if (d->kind != PKV_DECODE && !d->qo_indptr)
        return fail(PKV_ERR_INVALID_ARG, "prefill plans need qo_indptr");
    if (d->num_qo_heads <= 0 || d->num_kv_heads <= 0)
        return fail(PKV_ERR_INVALID_ARG, "head counts must be positive (%d, %d)", d->num_qo_heads,
                    d->num_kv_heads);
    if (d->num_qo_heads % d->num_kv_heads != 0)
        return fail(PKV_ERR_UNSUPPORTED, "num_qo_heads %d is not a multiple of num_kv_heads %d",
                    d->num_qo_heads, d->num_kv_heads);
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", d->head_dim);
    if (!ragged && d->page_size <= 0)
        return fail(PKV_ERR_INVALID_ARG, "page_size %d <= 0", d->page_size);
    if (d->num_pages < 0)
        return fail(PKV_ERR_INVALID_ARG, "num_pages %d < 0", d->num_pages);
    if (d->dtype != PKV_BF16)
        return fail(PKV_ERR_UNSUPPORTED, "dtype %d: only PKV_BF16 q/out are supported", d->dtype);
    if (d->kv_dtype != PKV_BF16 && d->kv_dtype != PKV_FP8_E4M3 && d->kv_dtype != PKV_FP8_E5M2)
        return fail(PKV_ERR_INVALID_ARG, "kv_dtype %d is not PKV_BF16, PKV_FP8_E4M3 or PKV_FP8_E5M2",
                    d->kv_dtype);
    if (d->kv_dtype != PKV_BF16 && d->kind == PKV_PREFILL_RAGGED)
        return fail(PKV_ERR_UNSUPPORTED, "8-bit K/V are supported in paged caches only");
    if (!(d->sm_scale == d->sm_scale) || std::isinf(d->sm_scale))
        return fail(PKV_ERR_INVALID_ARG, "sm_scale is not finite");
    if (!(d->sm_scale > 0.f))
        return fail(PKV_ERR_UNSUPPORTED, "sm_scale must be positive");
    for (float x : {d->logits_soft_cap, d->k_scale, d->v_scale})
        if (!(x == x) || std::isinf(x))
            return fail(PKV_ERR_INVALID_ARG, "logits_soft_cap, k_scale and v_scale must be finite");
    if (d->kind != PKV_DECODE &&
        d->num_qo_heads / d->num_kv_heads > kPrefillRows)
        return fail(PKV_ERR_UNSUPPORTED, "query-head group %d exceeds %d",
                    d->num_qo_heads / d->num_kv_heads, kPrefillRows);
    if (d->kv_indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "kv_indptr[0] = %d, expected 0", d->kv_indptr[0]);
    if (d->kind != PKV_DECODE && d->qo_indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "qo_indptr[0] = %d, expected 0", d->qo_indptr[0]);
    if (!ragged && B > 0 && d->kv_indptr[B] > 0 && !d->kv_indices)
        return fail(PKV_ERR_INVALID_ARG, "kv_indices is NULL but the batch holds pages");
    reqs.resize(B);
    for (int b = 0; b < B; ++b) {
        int64_t np = (int64_t)d->kv_indptr[b + 1] - d->kv_indptr[b];
        if (np < 0)
            return fail(PKV_ERR_INVALID_ARG, "kv_indptr decreases at request %d", b);
        int64_t kv_len = np;  // ragged: kv_indptr counts tokens
        if (!ragged) {
            int64_t last = d->kv_last_page_len[b];
            if (np > 0 && (last < 1 || last > d->page_size))
                return fail(PKV_ERR_INVALID_ARG, "kv_last_page_len[%d] = %lld outside [1, %d]", b,
                            (long long)last, d->page_size);
            kv_len = np > 0 ? (np - 1) * d->page_size + last : 0;
        }
        if (kv_len > INT32_MAX / 2)
            return fail(PKV_ERR_UNSUPPORTED, "request %d holds %lld tokens", b, (long long)kv_len);
        int64_t qo_begin, qo_len;
        if (d->kind != PKV_DECODE) {
            qo_begin = d->qo_indptr[b];
            qo_len = (int64_t)d->qo_indptr[b + 1] - d->qo_indptr[b];
            if (qo_len < 0)
                return fail(PKV_ERR_INVALID_ARG, "qo_indptr decreases at request %d", b);
        } else {
            qo_begin = b;
            qo_len = 1;
        }
        int64_t q_start = d->q_start ? (int64_t)d->q_start[b] : kv_len - qo_len;
        if (std::llabs(q_start) > INT32_MAX / 2)
            return fail(PKV_ERR_INVALID_ARG, "q_start[%d] out of range", b);
        reqs[b] = {qo_begin, qo_len, kv_len, (int64_t)d->kv_indptr[b], q_start};
    }
    return PKV_OK;
}

// Visible key interval [lo, hi] (inclusive; empty when hi < lo) of the query
// positions [p_min, p_max] taken together, for a request of kv_len keys.
void visible_interval(int64_t p_min, int64_t p_max, int64_t kv_len, int window_left, bool causal,
                      int64_t &lo, int64_t &hi)
{
    lo = window_left >= 0 ? std::max<int64_t>(0, p_min - window_left) : 0;
    hi = causal ? std::min<int64_t>(kv_len - 1, p_max) : kv_len - 1;
}

// Greedy longest-first assignment of item costs to `slots` equal workers; returns
// the finishing time of the busiest worker.
double simulate_makespan(std::vector<double> costs, int slots)
{
    std::sort(costs.begin(), costs.end(), std::greater<double>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < slots; ++i)
        load.push(0.0);
    for (double c : costs) {
        double t = load.top();
        load.pop();
        load.push(t + c);
    }
    double mx = 0;
    while (!load.empty()) {
        mx = std::max(mx, load.top());
        load.pop();
    }
    return mx;
}

int device_sm_count(int device)
{
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
        n = 148;
    return n;
}

// Decode: pick the KV tokens per split. A pure function of the plan inputs and the
// SM count: every candidate split size (no split first, then from 256 tokens up
// in steps of 1.25x) is scored by a simulated longest-first makespan of its CTAs
// over the SM slots (each CTA costing its tokens plus a fixed start-up cost, plus
// the partial-state traffic when split) plus a fixed cost for the merge pass
// when any request splits; a candidate must beat the best so far by 2% to win,
// which keeps splits rare unless they clearly pay (measured on GB300: a second
// pass and many short CTAs cost more than the tail they remove on 64-request
// batches).
int64_t choose_decode_chunk(const std::vector<int64_t> &lens, int head_blocks, int sms,
                            int ctas_per_sm)
{
    int64_t max_len = 0;
    for (int64_t l : lens)
        max_len = std::max(max_len, l);
    if (max_len <= 256)
        return std::max<int64_t>(max_len, 1);
    const int slots = sms * ctas_per_sm;
    const double kCtaOverhead = 96.0;   // token-row equivalents per CTA
    const double kPartialCost = 32.0;   // token-row equivalents per partial (write + merge read)
    const double kMergeFixed = 512.0;   // the merge pass (launch and drain), per slot
    std::vector<int64_t> cands{max_len};
    for (int64_t c = 256; c < max_len; c = round_up((int64_t)(c * 1.25), 64))
        cands.push_back(c);
    int64_t best_chunk = max_len;
    double best = 0;
    bool have = false;
    for (int64_t chunk : cands) {
        std::vector<double> costs;
        costs.reserve(lens.size() * 8);
        double merge = 0;
        bool any_split = false;
        for (int64_t l : lens) {
            if (l <= 0) {
                costs.push_back(kCtaOverhead);
                continue;
            }
            int64_t n = (l + chunk - 1) / chunk;
            int64_t per = round_up((l + n - 1) / n, 16);
            for (int64_t s = 0; s < n; ++s) {
                int64_t t = std::min(per, l - s * per);
                if (t <= 0)
                    break;
                for (int h = 0; h < head_blocks; ++h)
                    costs.push_back((double)t + kCtaOverhead + (n > 1 ? kPartialCost : 0.0));
            }
            if (n > 1) {
                merge += (double)n * head_blocks * kPartialCost / slots;
                any_split = true;
            }
        }
        double score = simulate_makespan(costs, slots) + merge + (any_split ? kMergeFixed : 0.0);
        if (!have || score < best * 0.98) {
            best = score;
            best_chunk = chunk;
            have = true;
        }
    }
    return best_chunk;
}

}  // namespace

namespace {

// The work schedule of a batch, built on the host from the host arrays alone.
struct Schedule {
    std::vector<RequestInfo> reqs;
    std::vector<PrefillItem> p_items;
    std::vector<DecodeItem> d_items;
    std::vector<int32_t> cta_items;  // prefill: list offsets (lists + 1 entries)
    int num_partials = 0;
    int num_counters = 0;
    int mask_mode = kMaskNone;
    int decode_tile = 64;
    int64_t total_q = 0;
};

// Splits per request that a capturable decode plan's workspace holds.
constexpr int kCapturableMaxSplits = 4;

// capturable: one prefill list per SM and at most kCapturableMaxSplits decode splits
// per request; fixed_tile > 0: the decode tile to use (a captured launch's variant).
void build_schedule(const pkv_plan_desc &d, const std::vector<HostRequest> &reqs, int device, bool capturable,
                    int fixed_tile, Schedule &sc)
{
    const int B = d.batch_size;
    const int group = d.num_qo_heads / d.num_kv_heads;
    const bool causal = d.causal != 0;
    const int W = d.window_left < 0 ? -1 : d.window_left;
    std::vector<RequestInfo> &h_reqs = sc.reqs;
    h_reqs.assign(B, RequestInfo{});
    int64_t total_q = 0;
    for (int b = 0; b < B; ++b) {
        const HostRequest &r = reqs[b];
        h_reqs[b] = {(int32_t)r.qo_begin, (int32_t)r.qo_len, (int32_t)r.kv_len,
                     (int32_t)r.kv_page_begin, (int32_t)r.q_start, 0, 0, 0};
        total_q = std::max<int64_t>(total_q, r.qo_begin + r.qo_len);
    }

    std::vector<PrefillItem> &p_items = sc.p_items;
    std::vector<DecodeItem> &d_items = sc.d_items;
    std::vector<int32_t> &cta_items = sc.cta_items;  // prefill: per-list item offsets
    int decode_tile = 64;
    int num_partials = 0;
    int num_counters = 0;
    int mask_mode = causal ? (W >= 0 ? kMaskCausalWindow : kMaskCausal)
                           : (W >= 0 ? kMaskWindow : kMaskNone);

    if (d.kind != PKV_DECODE) {
        const int T = prefill_kv_tile(d.head_dim);
        const int tq = prefill_tokens_per_cta(d.head_dim, group);
        // Ragged K/V: a TMA box may start at any row. Pages: at a page (TMA page
        // boxes) or anywhere (cp.async gathers).
        // 8-bit caches are gathered row by row.
        const int64_t kv_align = d.kind == PKV_PREFILL_RAGGED || d.kv_dtype != PKV_BF16 ? 1
                                 : prefill_pp_tma_page_size(d.page_size, d.head_dim)    ? std::min(d.page_size, T)
                                                                                        : 1;
        for (int b = 0; b < B; ++b) {
            const HostRequest &r = reqs[b];
            for (int64_t t0 = 0; t0 < r.qo_len; t0 += tq) {
                int64_t nt = std::min<int64_t>(tq, r.qo_len - t0);
                int64_t lo, hi;
                visible_interval(r.q_start + t0, r.q_start + t0 + nt - 1, r.kv_len, W, causal, lo, hi);
                // The item's KV tiles start at its first visible key, rounded down
                // only as far as the loader needs (a page for TMA page boxes), not
                // to a multiple of the tile: the window then spans the fewest tiles.
                int32_t start = 0, ntl = 0;
                if (hi >= lo) {
                    start = (int32_t)(lo / kv_align * kv_align);
                    ntl = (int32_t)((hi - start) / T + 1);
                }
                // Start tile: the query block's index times the golden ratio,
                // modulo the tile count, so that neighbouring blocks (which run at
                // the same time over nearly the same KV tiles) start far apart.
                const double frac = std::fmod((double)(t0 / tq) * 0.6180339887498949, 1.0);
                const int32_t rot = ntl > 1 ? std::min<int32_t>(ntl - 1, (int32_t)(frac * ntl)) : 0;
                for (int hk = 0; hk < d.num_kv_heads; ++hk)
                    p_items.push_back({b, hk, (int32_t)t0, (int32_t)nt, start, ntl, rot, 0});
            }
        }
        // Persistent CTAs, one per SM: longest-processing-time-first assignment of
        // the items to the least loaded CTA. Cost of an item in KV-tile steps: a
        // single query tile runs its softmax-bound chain alone (about 0.8 of the
        // two-tile ping-pong step, as measured through the schedule it yields),
        // plus a fixed cost per item (pipeline fill and epilogue).
        const int tq_tile = std::max(1, kPrefillRows / group);
        auto cost = [&](const PrefillItem &it) {
            const int nq = (d.head_dim <= 128 && it.ntok > tq_tile) ? 2 : 1;
            return it.kv_tiles * (nq == 2 ? 1.0 : 0.8) + 1.5;
        };
        std::stable_sort(p_items.begin(), p_items.end(),
                         [&](const PrefillItem &a, const PrefillItem &b) { return cost(a) > cost(b); });
        const int n_sm = device_sm_count(device);
        // A capturable plan keeps one list per SM (some may be empty): the launch's
        // grid is fixed when it is captured.
        const int G = capturable ? n_sm : (int)std::min<size_t>(p_items.size(), (size_t)n_sm);
        std::vector<std::vector<PrefillItem>> per_cta(G);
        std::priority_queue<std::pair<double, int>, std::vector<std::pair<double, int>>,
                            std::greater<std::pair<double, int>>>
            heap;
        for (int c = 0; c < G; ++c)
            heap.push({0.0, c});
        for (const PrefillItem &it : p_items) {
            auto [load, c] = heap.top();
            heap.pop();
            per_cta[c].push_back(it);
            heap.push({load + cost(it), c});
        }
        p_items.clear();
        cta_items.assign(1, 0);
        for (int c = 0; c < G; ++c) {
            p_items.insert(p_items.end(), per_cta[c].begin(), per_cta[c].end());
            cta_items.push_back((int32_t)p_items.size());
        }
    } else {
        const int head_blocks = (group + kDecodeRows - 1) / kDecodeRows;
        std::vector<int64_t> lens(B), los(B);
        for (int b = 0; b < B; ++b) {
            int64_t lo, hi;
            const HostRequest &r = reqs[b];
            visible_interval(r.q_start, r.q_start, r.kv_len, W, causal, lo, hi);
            los[b] = lo;
            lens[b] = std::max<int64_t>(0, hi - lo + 1);
        }
        int64_t chunk;
        if (d.disable_split_kv) {
            chunk = INT32_MAX;
        } else if (d.fixed_split_size > 0) {
            chunk = d.fixed_split_size;
        } else {
            const int ctas_per_sm = d.head_dim <= 128 ? 2 : 1;
            chunk = choose_decode_chunk(lens, head_blocks * d.num_kv_heads,
                                        device_sm_count(device), ctas_per_sm);
        }
        for (int b = 0; b < B; ++b) {
            int64_t L = lens[b];
            int64_t n = L > 0 ? (L + chunk - 1) / chunk : 1;
            int64_t per = L > 0 ? (d.fixed_split_size > 0 && !d.disable_split_kv
                                       ? chunk
                                       : round_up((L + n - 1) / n, 16))
                                : 0;
            if (L > 0)
                n = (L + per - 1) / per;
            if (capturable && n > kCapturableMaxSplits) {
                // the workspace of a capturable plan holds this many splits per request
                n = kCapturableMaxSplits;
                per = round_up((L + n - 1) / n, 16);
                n = (L + per - 1) / per;
            }
            int32_t pbase = -1, cbase = -1;
            if (n > 1) {
                pbase = num_partials;
                num_partials += (int32_t)n;
                cbase = num_counters;  // one arrival counter per (KV head, head block)
                num_counters += d.num_kv_heads * head_blocks;
            }
            for (int64_t s = 0; s < n; ++s) {
                int64_t j0 = los[b] + s * per;
                int64_t j1 = L > 0 ? std::min(los[b] + L, j0 + per) : j0;
                for (int hk = 0; hk < d.num_kv_heads; ++hk)
                    for (int h0 = 0; h0 < group; h0 += kDecodeRows)
                        d_items.push_back({b, hk, hk * group + h0, std::min(kDecodeRows, group - h0),
                                           (int32_t)j0, (int32_t)j1, n > 1 ? (int32_t)(pbase + s) : -1,
                                           pbase, (int32_t)n,
                                           n > 1 ? cbase + hk * head_blocks + h0 / kDecodeRows : -1,
                                           h_reqs[b].qo_begin, h_reqs[b].kv_len, h_reqs[b].kv_page_begin, 0});
            }
        }
        std::stable_sort(d_items.begin(), d_items.end(), [](const DecodeItem &a, const DecodeItem &b) {
            return (a.j1 - a.j0) > (b.j1 - b.j0);
        });
        decode_tile = fixed_tile > 0 ? fixed_tile
                                     : decode_tile_for(d.head_dim,
                                                       d_items.empty() ? 0 : d_items.front().j1 - d_items.front().j0,
                                                       (int64_t)d_items.size(), device_sm_count(device));
    }
    sc.num_partials = num_partials;
    sc.num_counters = num_counters;
    sc.mask_mode = mask_mode;
    sc.decode_tile = decode_tile;
    sc.total_q = total_q;

}

// Sizes of a plan's device workspace: the live schedule for an ordinary plan, the
// declared capacity for a capturable one.
struct Caps {
    int64_t batch = 0, total_q = 0, items = 0, lists = 0, partials = 0, counters = 0;
};

Caps caps_of(const pkv_plan_desc &d, const Schedule &sc)
{
    Caps c;
    c.batch = d.batch_size;
    c.total_q = sc.total_q;
    c.items = d.kind != PKV_DECODE ? (int64_t)sc.p_items.size() : (int64_t)sc.d_items.size();
    c.lists = sc.cta_items.empty() ? 0 : (int64_t)sc.cta_items.size() - 1;
    c.partials = sc.num_partials;
    c.counters = sc.num_counters;
    return c;
}

Caps caps_for_capacity(const pkv_plan_desc &d, const pkv_plan_caps &cap, int n_sm)
{
    const int group = d.num_qo_heads / d.num_kv_heads;
    Caps c;
    c.batch = cap.max_batch;
    if (d.kind != PKV_DECODE) {
        const int64_t tq = prefill_tokens_per_cta(d.head_dim, group);
        c.total_q = cap.max_total_q;
        c.items = (int64_t)d.num_kv_heads * ((cap.max_total_q + tq - 1) / tq + cap.max_batch);
        c.lists = n_sm;
    } else {
        const int64_t head_blocks = (group + kDecodeRows - 1) / kDecodeRows;
        c.total_q = cap.max_batch;
        c.items = (int64_t)cap.max_batch * d.num_kv_heads * head_blocks * kCapturableMaxSplits;
        c.partials = (int64_t)cap.max_batch * kCapturableMaxSplits;
        c.counters = (int64_t)cap.max_batch * d.num_kv_heads * head_blocks;
    }
    return c;
}

// requests | items | list offsets | live item count (uploaded) | partial o | partial
// lse | arrival counters | status.
struct Layout {
    size_t reqs, items, cta, live, po, pl, cnt, status, bytes, upload;
};

Layout layout_for(const pkv_plan_desc &d, const Caps &c)
{
    const size_t item_bytes = d.kind != PKV_DECODE ? sizeof(PrefillItem) : sizeof(DecodeItem);
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        size_t at = off;
        off = (size_t)round_up((int64_t)(off + bytes), 256);
        return at;
    };
    Layout l{};
    l.reqs = carve(sizeof(RequestInfo) * std::max<int64_t>(1, c.batch));
    l.items = carve(item_bytes * std::max<int64_t>(1, c.items));
    l.cta = carve(sizeof(int32_t) * (std::max<int64_t>(0, c.lists) + 1));
    l.live = carve(sizeof(int32_t) * 4);
    l.po = carve(sizeof(float) * (size_t)c.partials * d.num_qo_heads * d.head_dim);
    l.pl = carve(sizeof(float) * (size_t)c.partials * d.num_qo_heads);
    l.cnt = carve(sizeof(int32_t) * std::max<int64_t>(1, c.counters));
    l.status = carve(sizeof(int32_t) * 4);
    l.bytes = off;
    l.upload = l.po;
    return l;
}

// The uploaded part of the workspace image of a schedule.
void fill_image(const pkv_plan_desc &d, const Schedule &sc, const Layout &l, uint8_t *img)
{
    std::memset(img, 0, l.upload);
    std::memcpy(img + l.reqs, sc.reqs.data(), sizeof(RequestInfo) * sc.reqs.size());
    if (d.kind != PKV_DECODE)
        std::memcpy(img + l.items, sc.p_items.data(), sizeof(PrefillItem) * sc.p_items.size());
    else
        std::memcpy(img + l.items, sc.d_items.data(), sizeof(DecodeItem) * sc.d_items.size());
    std::memcpy(img + l.cta, sc.cta_items.data(), sizeof(int32_t) * sc.cta_items.size());
    const int32_t live = d.kind != PKV_DECODE ? (int32_t)sc.p_items.size() : (int32_t)sc.d_items.size();
    std::memcpy(img + l.live, &live, sizeof(live));
}

}  // namespace

extern "C" {

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_OOM: return "PKV_ERR_OOM";
    case PKV_ERR_DEVICE_BOUNDS: return "PKV_ERR_DEVICE_BOUNDS";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    default: return "PKV_ERR_UNKNOWN";
    }
}

const char *pkv_last_error(void) { return g_last_error.c_str(); }

int pkv_abi_version(void) { return PKV_ABI_VERSION; }

namespace {

int create_plan(pkv_plan **out, const pkv_plan_desc *desc, const pkv_plan_caps *capacity, void *stream_)
{
    g_last_error.clear();
    if (!out)
        return fail(PKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    std::vector<HostRequest> reqs;
    int st = validate(desc, reqs);
    if (st != PKV_OK)
        return st;
    const pkv_plan_desc &d = *desc;
    const bool capturable = capacity != nullptr;
    if (capturable && d.kind == PKV_PREFILL_RAGGED)
        return fail(PKV_ERR_UNSUPPORTED, "ragged plans are not capturable (the K/V row count is baked into a launch)");
    if (capturable && (capacity->max_batch < d.batch_size || capacity->max_batch < 1 ||
                       (d.kind != PKV_DECODE && capacity->max_total_q < 1)))
        return fail(PKV_ERR_INVALID_ARG, "capacity: max_batch must be >= 1 and >= batch_size%s",
                    d.kind != PKV_DECODE ? ", max_total_q >= 1" : "");
    cudaStream_t stream = (cudaStream_t)stream_;
    int device = 0;
    cudaError_t ce = cudaGetDevice(&device);
    if (ce != cudaSuccess)
        return cuda_fail(ce, "cudaGetDevice");
    const int n_sm = device_sm_count(device);

    Schedule sc;
    build_schedule(d, reqs, device, capturable, 0, sc);
    const Caps caps = capturable ? caps_for_capacity(d, *capacity, n_sm) : caps_of(d, sc);
    if (capturable && (sc.total_q > caps.total_q))
        return fail(PKV_ERR_UNSUPPORTED, "the batch has %lld query rows, the capacity %lld",
                    (long long)sc.total_q, (long long)caps.total_q);
    const Layout lay = layout_for(d, caps);

    pkv_plan *plan = new (std::nothrow) pkv_plan();
    if (!plan)
        return fail(PKV_ERR_OOM, "host allocation of the plan failed");
    ce = cudaMalloc(&plan->workspace, lay.bytes);
    if (ce != cudaSuccess) {
        delete plan;
        return cuda_fail(ce, "cudaMalloc(plan workspace)");
    }
    std::vector<uint8_t> image(lay.upload, 0);
    fill_image(d, sc, lay, image.data());
    uint8_t *base = (uint8_t *)plan->workspace;
    ce = cudaMemcpyAsync(base, image.data(), lay.upload, cudaMemcpyHostToDevice, stream);
    if (ce == cudaSuccess)
        ce = cudaMemsetAsync(base + lay.status, 0, sizeof(int32_t) * 4, stream);
    if (ce == cudaSuccess)  // arrival counters start at zero; each merge resets its own
        ce = cudaMemsetAsync(base + lay.cnt, 0, lay.status - lay.cnt, stream);
    if (ce == cudaSuccess)
        ce = cudaStreamSynchronize(stream);  // the host image is freed on return
    if (ce == cudaSuccess && capturable) {
        for (int k = 0; k < 2 && ce == cudaSuccess; ++k) {
            ce = cudaHostAlloc(&plan->staging[k], lay.upload, cudaHostAllocDefault);
            if (ce == cudaSuccess)
                ce = cudaEventCreateWithFlags(&plan->staging_done[k], cudaEventDisableTiming);
        }
    }
    if (ce != cudaSuccess) {
        for (int k = 0; k < 2; ++k) {
            if (plan->staging[k])
                cudaFreeHost(plan->staging[k]);
            if (plan->staging_done[k])
                cudaEventDestroy(plan->staging_done[k]);
        }
        cudaFree(plan->workspace);
        delete plan;
        return cuda_fail(ce, "uploading the plan");
    }
    plan->desc = d;
    plan->desc.qo_indptr = plan->desc.kv_indptr = plan->desc.kv_last_page_len = nullptr;
    plan->desc.q_start = nullptr;
    plan->desc.window_left = d.window_left < 0 ? -1 : d.window_left;
    plan->device = device;
    plan->n_sm = n_sm;
    plan->capturable = capturable;
    plan->mask_mode = sc.mask_mode;
    plan->num_items = (int)(d.kind != PKV_DECODE ? sc.p_items.size() : sc.d_items.size());
    plan->num_partials = sc.num_partials;
    plan->num_ctas = sc.cta_items.empty() ? 0 : (int)sc.cta_items.size() - 1;
    plan->decode_tile = sc.decode_tile;
    plan->total_q = sc.total_q;
    plan->total_kv = d.batch_size > 0 ? d.kv_indptr[d.batch_size] : 0;
    plan->cap_items = caps.items;
    plan->cap_total_q = caps.total_q;
    plan->cap_batch = caps.batch;
    plan->upload_bytes = lay.upload;
    plan->kv_indices = d.kv_indices;
    plan->workspace_bytes = lay.bytes;
    plan->d_reqs = (RequestInfo *)(base + lay.reqs);
    plan->d_items = base + lay.items;
    plan->d_cta_items = (int32_t *)(base + lay.cta);
    plan->d_live = (int32_t *)(base + lay.live);
    plan->d_partial_o = (float *)(base + lay.po);
    plan->d_partial_lse = (float *)(base + lay.pl);
    plan->d_status = (int32_t *)(base + lay.status);
    plan->d_counters = (int32_t *)(base + lay.cnt);
    *out = plan;
    return PKV_OK;
}

}  // namespace

int pkv_plan_create(pkv_plan **out, const pkv_plan_desc *desc, void *stream)
{
    NvtxRange range("pkv_plan_create");
    return create_plan(out, desc, nullptr, stream);
}

int pkv_plan_create_capturable(pkv_plan **out, const pkv_plan_desc *desc, const pkv_plan_caps *caps,
                               void *stream)
{
    NvtxRange range("pkv_plan_create_capturable");
    if (!caps) {
        g_last_error.clear();
        if (out)
            *out = nullptr;
        return fail(PKV_ERR_INVALID_ARG, "caps is NULL");
    }
    return create_plan(out, desc, caps, stream);
}

int pkv_plan_update(pkv_plan *plan, const pkv_plan_desc *desc, void *stream_)
{
    NvtxRange range("pkv_plan_update");
    g_last_error.clear();
    if (!plan)
        return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
    if (!plan->capturable)
        return fail(PKV_ERR_INVALID_ARG, "pkv_plan_update needs a plan from pkv_plan_create_capturable");
    std::vector<HostRequest> reqs;
    int st = validate(desc, reqs);
    if (st != PKV_OK)
        return st;
    const pkv_plan_desc &d = *desc, &o = plan->desc;
    const int W = d.window_left < 0 ? -1 : d.window_left;
    // What the captured launches bake in must not change.
    if (d.kind != o.kind || d.num_qo_heads != o.num_qo_heads || d.num_kv_heads != o.num_kv_heads ||
        d.head_dim != o.head_dim || d.page_size != o.page_size || W != o.window_left ||
        (d.causal != 0) != (o.causal != 0) || d.sm_scale != o.sm_scale || d.dtype != o.dtype ||
        d.logits_soft_cap != o.logits_soft_cap || d.k_scale != o.k_scale || d.v_scale != o.v_scale ||
        d.kv_dtype != o.kv_dtype || d.wait_limit_us != o.wait_limit_us || d.wait_probe != o.wait_probe ||
        d.num_pages != o.num_pages || d.kv_indices != o.kv_indices)
        return fail(PKV_ERR_INVALID_ARG,
                    "update must keep kind, heads, head_dim, page_size, window_left, causal, sm_scale, "
                    "dtype, kv_dtype, soft cap, scales, wait bound and probe, num_pages and the kv_indices "
                    "pointer of the plan");
    if (d.batch_size > plan->cap_batch)
        return fail(PKV_ERR_UNSUPPORTED, "batch %d exceeds the plan's capacity %lld", d.batch_size,
                    (long long)plan->cap_batch);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != plan->device)
        return fail(PKV_ERR_INVALID_ARG, "plan was made on device %d, current device is %d", plan->device, cur);
    Schedule sc;
    build_schedule(d, reqs, plan->device, true, plan->decode_tile, sc);
    const int64_t items = d.kind != PKV_DECODE ? (int64_t)sc.p_items.size() : (int64_t)sc.d_items.size();
    if (sc.total_q > plan->cap_total_q || items > plan->cap_items)
        return fail(PKV_ERR_UNSUPPORTED, "the batch needs %lld query rows and %lld work items, the capacity is %lld "
                    "and %lld", (long long)sc.total_q, (long long)items, (long long)plan->cap_total_q,
                    (long long)plan->cap_items);
    pkv_plan_caps cap{};
    cap.max_batch = (int32_t)plan->cap_batch;
    cap.max_total_q = plan->cap_total_q;
    const Layout lay = layout_for(plan->desc, caps_for_capacity(plan->desc, cap, plan->n_sm));
    cudaStream_t stream = (cudaStream_t)stream_;
    // Two pinned staging images, each reused only once its previous upload is done
    // (an event wait that is normally already satisfied; nothing else waits).
    const int k = plan->staging_next;
    cudaError_t ce = cudaEventSynchronize(plan->staging_done[k]);
    if (ce != cudaSuccess)
        return cuda_fail(ce, "waiting for the staging image");
    fill_image(plan->desc, sc, lay, (uint8_t *)plan->staging[k]);
    ce = cudaMemcpyAsync(plan->workspace, plan->staging[k], lay.upload, cudaMemcpyHostToDevice, stream);
    if (ce == cudaSuccess)
        ce = cudaEventRecord(plan->staging_done[k], stream);
    if (ce != cudaSuccess)
        return cuda_fail(ce, "uploading the updated plan");
    plan->staging_next = k ^ 1;
    plan->num_items = (int)items;
    plan->num_partials = sc.num_partials;
    plan->num_ctas = sc.cta_items.empty() ? 0 : (int)sc.cta_items.size() - 1;
    plan->total_q = sc.total_q;
    plan->desc.batch_size = d.batch_size;
    plan->desc.fixed_split_size = d.fixed_split_size;
    plan->desc.disable_split_kv = d.disable_split_kv;
    return PKV_OK;
}

int pkv_plan_destroy(pkv_plan *plan)
{
    if (!plan)
        return PKV_OK;
    for (int k = 0; k < 2; ++k) {
        if (plan->staging_done[k]) {
            cudaEventSynchronize(plan->staging_done[k]);
            cudaEventDestroy(plan->staging_done[k]);
        }
        if (plan->staging[k])
            cudaFreeHost(plan->staging[k]);
    }
    cudaError_t ce = cudaFree(plan->workspace);
    delete plan;
    if (ce != cudaSuccess)
        return cuda_fail(ce, "cudaFree(plan workspace)");
    return PKV_OK;
}

int pkv_plan_get_info(const pkv_plan *plan, pkv_plan_info *info)
{
    if (!plan || !info)
        return fail(PKV_ERR_INVALID_ARG, "plan and info are required");
    std::memset(info, 0, sizeof *info);
    info->kind = plan->desc.kind;
    info->num_work_items = plan->num_items;
    info->num_partials = plan->num_partials;
    info->mask_mode = plan->mask_mode;
    info->workspace_bytes = (int64_t)plan->workspace_bytes;
    info->total_q = plan->total_q;
    info->kernels_per_run = (plan->num_items > 0 || plan->capturable) ? 1 : 0;
    info->kv_tile = plan->desc.kind == PKV_DECODE
                        ? decode_kernel_tile(plan->decode_tile, plan->desc.head_dim, plan->desc.kv_dtype)
                        : prefill_kv_tile(plan->desc.head_dim);
    return PKV_OK;
}

int pkv_plan_set_timing_events(pkv_plan *plan, void *ev_begin, void *ev_end)
{
    if (!plan)
        return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
    plan->ev_begin = (cudaEvent_t)ev_begin;
    plan->ev_end = (cudaEvent_t)ev_end;
    return PKV_OK;
}

int pkv_plan_device_status(const pkv_plan *plan, int32_t *status)
{
    if (!plan || !status)
        return fail(PKV_ERR_INVALID_ARG, "plan and status are required");
    int32_t h = 0;
    cudaError_t ce = cudaDeviceSynchronize();
    if (ce == cudaSuccess)
        ce = cudaMemcpy(&h, plan->d_status, sizeof h, cudaMemcpyDeviceToHost);
    if (ce == cudaSuccess)
        ce = cudaMemset(plan->d_status, 0, sizeof(int32_t));
    if (ce != cudaSuccess)
        return cuda_fail(ce, "reading the device status");
    *status = h;
    return PKV_OK;
}

static int page_shift_of(int page_size)
{
    if (page_size <= 0 || (page_size & (page_size - 1)))
        return -1;
    int s = 0;
    while ((1 << s) < page_size)
        ++s;
    return s;
}

static bool misaligned(const void *p, uintptr_t a) { return ((uintptr_t)p) % a != 0; }

int pkv_run(const pkv_plan *plan, const void *q, const void *k_cache, const void *v_cache, void *out,
            float *lse, void *stream_)
{
    NvtxRange range(plan && plan->desc.kind == PKV_DECODE ? "pkv_run decode" : "pkv_run prefill");
    g_last_error.clear();
    if (!plan)
        return fail(PKV_ERR_INVALID_ARG, "plan is NULL");
    if ((plan->total_q > 0 || plan->capturable) && (!q || !out))
        return fail(PKV_ERR_INVALID_ARG, "q and out are required");
    if ((plan->num_items > 0 || plan->capturable) && (!k_cache || !v_cache))
        return fail(PKV_ERR_INVALID_ARG, "k_cache and v_cache are required");
    if (misaligned(q, 16) || misaligned(k_cache, 16) || misaligned(v_cache, 16) ||
        misaligned(out, 16) || misaligned(lse, 4))
        return fail(PKV_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned, lse 4-byte");
    int cur = -1;
    if (cudaGetDevice(&cur) == cudaSuccess && cur != plan->device)
        return fail(PKV_ERR_INVALID_ARG, "plan was made on device %d, current device is %d",
                    plan->device, cur);
    // A capturable plan always launches (its launch may be captured and replayed
    // after pkv_plan_update); its decode grid is the capacity, its prefill grid one
    // CTA per SM, and CTAs without work leave at once.
    if (plan->num_items == 0 && !plan->capturable)
        return PKV_OK;
    cudaStream_t stream = (cudaStream_t)stream_;
    const pkv_plan_desc &d = plan->desc;
    cudaError_t ce;
    if (d.kind == PKV_DECODE) {
        DecodeParams p{};
        p.items = (const DecodeItem *)plan->d_items;
        p.reqs = plan->d_reqs;
        p.kv_indices = plan->kv_indices;
        p.q = (const uint16_t *)q;
        p.k_cache = (const uint16_t *)k_cache;
        p.v_cache = (const uint16_t *)v_cache;
        p.out = (uint16_t *)out;
        p.lse = lse;
        p.partial_o = plan->d_partial_o;
        p.partial_lse = plan->d_partial_lse;
        p.merge_counters = plan->d_counters;
        p.live_items = plan->capturable ? plan->d_live : nullptr;
        p.status = plan->d_status;
        p.num_qo_heads = d.num_qo_heads;
        p.num_kv_heads = d.num_kv_heads;
        p.page_size = d.page_size;
        p.page_shift = page_shift_of(d.page_size);
        p.num_pages = d.num_pages;
        const LogitFactors lf = logit_factors(d);
        p.sm_scale_log2 = lf.sm_scale_log2;
        p.cap_in = lf.cap_in;
        p.cap_out = lf.cap_out;
        p.v_scale = lf.v_scale;
        p.kv_dtype = d.kv_dtype;
        p.wait_probe = d.wait_probe;
        p.wait_ns = wait_ns_of(d);
        if (plan->ev_begin && (ce = cudaEventRecord(plan->ev_begin, stream)) != cudaSuccess)
            return cuda_fail(ce, "cudaEventRecord");
        ce = launch_decode(p, d.head_dim, plan->capturable ? (int)plan->cap_items : plan->num_items, stream,
                           plan->decode_tile);
        if (ce != cudaSuccess)
            return cuda_fail(ce, "decode kernel launch");
        if (plan->ev_end && (ce = cudaEventRecord(plan->ev_end, stream)) != cudaSuccess)
            return cuda_fail(ce, "cudaEventRecord");
        return PKV_OK;
    }
    PrefillParams p{};
    p.items = (const PrefillItem *)plan->d_items;
    p.cta_items = plan->d_cta_items;
    p.reqs = plan->d_reqs;
    p.kv_indices = plan->kv_indices;
    p.q = (const uint16_t *)q;
    p.k_cache = (const uint16_t *)k_cache;
    p.v_cache = (const uint16_t *)v_cache;
    p.out = (uint16_t *)out;
    p.lse = lse;
    p.status = plan->d_status;
    p.num_qo_heads = d.num_qo_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.group = d.num_qo_heads / d.num_kv_heads;
    p.tokens_per_tile = std::max(1, kPrefillRows / p.group);
    p.total_q = (int32_t)(plan->capturable ? plan->cap_total_q : plan->total_q);
    p.page_size = d.page_size;
    p.page_shift = page_shift_of(d.page_size);
    p.num_pages = d.num_pages;
    p.window_left = d.window_left;
    const LogitFactors lf = logit_factors(d);
    p.sm_scale_log2 = lf.sm_scale_log2;
    p.cap_in = lf.cap_in;
    p.cap_out = lf.cap_out;
    p.v_scale = lf.v_scale;
    p.ragged = d.kind == PKV_PREFILL_RAGGED ? 1 : 0;
    p.kv_dtype = d.kv_dtype;
    p.wait_probe = d.wait_probe;
    p.wait_ns = wait_ns_of(d);
    p.total_kv = (int32_t)plan->total_kv;
    if (p.ragged) {
        p.page_size = 1;
        p.page_shift = 0;
        p.num_pages = (int32_t)plan->total_kv;
    }
    if (plan->ev_begin && (ce = cudaEventRecord(plan->ev_begin, stream)) != cudaSuccess)
        return cuda_fail(ce, "cudaEventRecord");
    ce = launch_prefill_pp(p, d.head_dim, plan->mask_mode, plan->capturable ? plan->n_sm : plan->num_ctas, stream);
    if (ce != cudaSuccess)
        return cuda_fail(ce, "prefill kernel launch");
    if (plan->ev_end && (ce = cudaEventRecord(plan->ev_end, stream)) != cudaSuccess)
        return cuda_fail(ce, "cudaEventRecord");
    return PKV_OK;
}

int pkv_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b, void *v_out,
                    float *s_out, int64_t n_tokens, int32_t n_heads, int32_t head_dim, int32_t dtype,
                    void *stream)
{
    NvtxRange range("pkv_merge_state");
    g_last_error.clear();
    if (n_tokens < 0 || n_heads < 0)
        return fail(PKV_ERR_INVALID_ARG, "negative size");
    if (dtype != PKV_BF16 && dtype != PKV_F32)
        return fail(PKV_ERR_UNSUPPORTED, "merge_state dtype %d", dtype);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", head_dim);
    const int64_t rows = n_tokens * (int64_t)n_heads;
    if (rows == 0)
        return PKV_OK;
    if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out)
        return fail(PKV_ERR_INVALID_ARG, "null pointer");
    if (misaligned(v_a, 16) || misaligned(v_b, 16) || misaligned(v_out, 16))
        return fail(PKV_ERR_INVALID_ARG, "value pointers must be 16-byte aligned");
    cudaError_t ce = launch_merge_state(v_a, s_a, v_b, s_b, v_out, s_out, rows, head_dim, dtype,
                                        (cudaStream_t)stream);
    if (ce != cudaSuccess)
        return cuda_fail(ce, "merge_state launch");
    return PKV_OK;
}

}  // extern "C"
