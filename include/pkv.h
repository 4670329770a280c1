/*
 * pkv.h - C ABI of libpkv: batched attention over a paged KV cache with a
 * per-element sliding-window mask, for NVIDIA GB300 (sm_103a).
 *
 * Semantics (what every entry point computes):
 *   For request b, query row i and query head h, the key at logical position j of
 *   the request's cache is visible iff
 *       (!causal || j <= p) && (window_left < 0 || j >= p - window_left),
 *   with p = q_start[b] + i (q_start defaults to kv_len_b - qo_len_b, so extend rows
 *   sit after the cached prefix). window_left = W therefore admits the W+1 keys
 *   [p-W, p] (the FlashInfer convention spelled out in AMD flashinfer PR #234, "Why
 *   each fix" 1; the mask k_abs >= q_abs - window of sglang flashinfer_backend.py,
 *   _build_swa_prefix_custom_mask), and any negative window_left means no window.
 *   out = softmax(sm_scale * q K^T over the visible keys) V, and
 *   lse = ln(sum over visible keys of exp(sm_scale * q.k)) (natural log of the
 *   scaled logits). A row with no visible key gets out = 0 and lse = -inf.
 *   Query head h reads KV head h / (num_qo_heads / num_kv_heads).
 *
 * Why the window lives in the plan: sglang PR #31501 ("Pass window_left at plan
 * time for the SWA paged prefill wrapper") fixed wrong outputs caused by a plan
 * made without the window and a run given one. Here window_left and causal are
 * plan arguments only; pkv_run takes neither, so the two cannot disagree.
 *
 * Layouts (all contiguous, row-major, "NHD" as in flashinfer_backend.py):
 *   q, out        : [total_q, num_qo_heads, head_dim] bf16
 *   lse           : [total_q, num_qo_heads] fp32
 *   k_cache/v_cache: [num_pages, page_size, num_kv_heads, head_dim] bf16
 *   Request b owns pages kv_indices[kv_indptr[b] .. kv_indptr[b+1]); its last page
 *   holds kv_last_page_len[b] in [1, page_size] valid slots, so
 *   kv_len_b = (kv_indptr[b+1] - kv_indptr[b] - 1) * page_size + kv_last_page_len[b]
 *   (0 when the request has no pages). The query rows of request b are
 *   qo_indptr[b] .. qo_indptr[b+1].
 *
 * Errors: every call returns a pkv_status; nothing traps or aborts. Invalid
 * arguments are rejected on the host before any launch (the "fail at plan() with a
 * clear message" pattern of AMD flashinfer PR #234 and flashinfer_backend.py's
 * plan-time asserts). pkv_last_error() gives a human-readable reason for the last
 * failure on the calling thread. Faults the host cannot see (a page id outside
 * [0, num_pages) in kv_indices) are recorded by the kernels in a device status
 * word instead of being dereferenced; read it with pkv_plan_device_status().
 *
 * Tracing: the host side of every entry point is an NVTX range named after it
 * ("pkv_run decode" / "pkv_run prefill" for runs), shown by profilers' timelines; with
 * no tool attached the range calls return at once.
 *
 * Threading and streams: a plan may be run from one host thread at a time; all
 * launches are asynchronous on the caller's stream (a cudaStream_t passed as void*,
 * NULL = legacy default stream). pkv_run and pkv_merge_state never synchronise;
 * pkv_plan_create waits for its own upload and pkv_plan_device_status for the
 * device.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 5

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* malformed argument (null, negative size, bad indptr) */
    PKV_ERR_UNSUPPORTED = 2,   /* well-formed but not supported (head_dim, dtype, ...) */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    PKV_ERR_OOM = 4,           /* device or host allocation failed */
    PKV_ERR_DEVICE_BOUNDS = 5, /* a kernel met a page id outside [0, num_pages) */
    PKV_ERR_TIMEOUT = 6        /* a bounded device wait gave up */
} pkv_status;

typedef enum pkv_kind {
    PKV_PREFILL = 0,        /* ragged query rows per request (extend over a cached prefix) */
    PKV_DECODE = 1,         /* exactly one query row per request */
    PKV_PREFILL_RAGGED = 2  /* ragged query rows against contiguous, non-paged K/V: k_cache
                               and v_cache passed to pkv_run are [total_kv, H_kv, d] with the
                               keys of request b at rows [kv_indptr[b], kv_indptr[b+1]);
                               kv_indptr counts tokens; kv_indices, kv_last_page_len,
                               page_size and num_pages are ignored (the ragged extend of
                               flashinfer_backend.py forward_extend, whose result is merged
                               with a paged prefix's by pkv_merge_state). Not capturable. */
} pkv_kind;

typedef enum pkv_dtype {
    PKV_BF16 = 0,
    PKV_F32 = 1,     /* merge_state values only */
    PKV_FP8_E4M3 = 2, /* 8-bit K/V caches (pkv_plan_desc.kv_dtype, paged plans): OCP E4M3,
                         torch.float8_e4m3fn */
    PKV_FP8_E5M2 = 3  /* OCP E5M2, torch.float8_e5m2 */
} pkv_dtype;

/*
 * Everything a plan needs to know. The fields mirror the arguments of the pages'
 * plan calls (flashinfer_backend.py: fast_prefill_plan's _cached_module.plan
 * arguments and call_begin_forward's begin_forward), with window_left and causal
 * fixed here and nowhere else (sglang PR #31501).
 */
typedef struct pkv_plan_desc {
    int32_t kind;                    /* pkv_kind */
    int32_t batch_size;              /* B >= 0 */
    const int32_t *qo_indptr;        /* HOST [B+1], non-decreasing from 0; PREFILL only
                                        (DECODE: NULL, one row per request) */
    const int32_t *kv_indptr;        /* HOST [B+1], non-decreasing from 0, in pages */
    const int32_t *kv_last_page_len; /* HOST [B], each in [1, page_size] (ignored for a
                                        request with no pages) */
    const int32_t *q_start;          /* HOST [B] or NULL: position of each request's
                                        first query row (NULL: kv_len - qo_len) */
    const int32_t *kv_indices;       /* DEVICE [kv_indptr[B]] physical page ids; BORROWED:
                                        must stay valid and unchanged until the last
                                        pkv_run of this plan */
    int32_t num_pages;               /* pages in k_cache / v_cache (bound for page ids) */
    int32_t num_qo_heads;
    int32_t num_kv_heads;            /* divides num_qo_heads */
    int32_t head_dim;                /* 64, 128 or 256 */
    int32_t page_size;               /* >= 1 */
    int32_t window_left;             /* W >= 0: keys [p-W, p]; < 0: no window */
    int32_t causal;                  /* nonzero: keys j <= p only */
    float sm_scale;                  /* logit scale, e.g. 1/sqrt(head_dim) */
    int32_t fixed_split_size;        /* DECODE: KV tokens per split (> 0), or <= 0 to
                                        let the plan choose */
    int32_t disable_split_kv;        /* nonzero: one pass per (request, KV head) */
    int32_t dtype;                   /* pkv_dtype of q, caches and out: PKV_BF16 */
    /* The per-layer arguments flashinfer_backend.py passes with every attention call
     * (forward_extend / forward_decode: the layer's logit soft cap, k_scale and
     * v_scale); the pages do not define them further, the readings taken are:
     *   logit_j = cap * tanh(sm_scale * k_scale * q.k_j / cap)   (cap > 0; <= 0: no cap)
     *   out = v_scale * sum_j softmax_j v_j                      (K, V dequantised)
     * A scale <= 0 means 1 (so a zero-initialised descriptor keeps the plain method). */
    float logits_soft_cap;
    float k_scale;
    float v_scale;
    /* Element type of k_cache and v_cache: PKV_BF16 (0), or an 8-bit float,
     * PKV_FP8_E4M3 or PKV_FP8_E5M2 (flashinfer_backend.py, should_use_tensor_core, names
     * torch.float8_e4m3fn and torch.float8_e5m2 as KV cache dtypes). The caches then
     * hold one byte per element in the same [num_pages, page_size, H_kv, d] layout,
     * K = k_scale * (stored value) and V = v_scale * (stored value); q and out stay
     * bf16. PREFILL_RAGGED plans take bf16 K/V only (PKV_ERR_UNSUPPORTED otherwise). */
    int32_t kv_dtype;
    /* Bound of every wait inside the kernels of this plan's runs, in microseconds;
     * <= 0 means the default of 2 s. A wait that runs out records PKV_ERR_TIMEOUT in
     * the plan's device status (pkv_plan_device_status), the kernel's other roles leave
     * at their next wait, the copies and tensor-core operations already issued are
     * waited for (each wait again bounded), and the kernel returns: a clear error
     * instead of a launch that never ends (the failure mode AMD flashinfer PR #234,
     * "Why each fix", turns into an error at plan time). */
    int32_t wait_limit_us;
    /* Test hook for the path above: nonzero makes the first wait of every CTA's
     * consuming role (decode: the compute warps' first K/V stage; prefill: the
     * tensor-core issuer's first K/V tile) wait on a barrier that nothing completes,
     * so that it runs out after wait_limit_us. Out and lse are then unspecified.
     * Leave 0 in normal use. */
    int32_t wait_probe;
} pkv_plan_desc;

typedef struct pkv_plan pkv_plan;

/* Facts about a plan, for tests and benchmarks. */
typedef struct pkv_plan_info {
    int32_t kind;
    int32_t num_work_items;    /* CTAs of the main kernel */
    int32_t num_partials;      /* split-KV partial states (0: no merge pass) */
    int32_t mask_mode;         /* 0 none, 1 causal, 2 causal + window, 3 window only */
    int64_t workspace_bytes;   /* device memory owned by the plan */
    int64_t total_q;           /* query rows */
    int32_t kernels_per_run;   /* launches issued by one pkv_run */
    int32_t kv_tile;           /* KV tokens per tile of the main kernel (decode: 32 or 64,
                                  64 or 128 over an 8-bit cache at head_dim <= 128;
                                  prefill: 128, or 64 at head_dim 256) */
} pkv_plan_info;

/*
 * pkv_plan_create: validate `desc`, decompose the batch into work items (request x
 * KV head x query tile for PREFILL; request x KV head x KV split for DECODE), each
 * with its KV tile range already clipped to [p_min - W, p_max], pick the mask
 * specialisation, and upload the work list to a device workspace that the plan
 * owns (cudaMalloc on the current device). The upload is issued on `stream` and
 * waited for before returning, so the plan is usable from any stream; nothing is
 * read back from the device (the schedule comes from the host arrays alone). Host
 * arrays are copied and may be freed on return.
 * Returns PKV_OK and sets *out, or an error with *out = NULL.
 */
PKV_API int pkv_plan_create(pkv_plan **out, const pkv_plan_desc *desc, void *stream);

/* Capacity of a capturable plan. */
typedef struct pkv_plan_caps {
    int32_t max_batch;    /* requests any later batch may hold (>= 1) */
    int32_t reserved;
    int64_t max_total_q;  /* PREFILL: query rows any later batch may hold (>= 1); q, out
                             and lse passed to pkv_run must hold this many rows. Ignored
                             for DECODE (one row per request). */
} pkv_plan_caps;

/*
 * pkv_plan_create_capturable: a plan whose pkv_run may be captured into a CUDA graph
 * once and replayed for later batches re-planned with pkv_plan_update. The launch
 * shapes are fixed by the capacity, not by the batch: the decode grid holds
 * max_batch x H_kv x ceil(group/16) x 4 CTAs (at most 4 KV splits per request) and
 * CTAs beyond the live work items return at once; prefill runs one persistent CTA per
 * SM whose work lists may be empty. The kernel variant (mask mode, decode KV tile,
 * TMA or cp.async gather) is chosen from this first batch and kept. This addresses
 * the baked-grid failure of a captured paged-attention launch described on the
 * AMD flashinfer PR #234 page ("Why each fix"), and the sync-free re-plan from host
 * metadata of flashinfer_backend.py's fast_prefill_plan.
 * Allocates the workspace for the capacity and two pinned staging images; the first
 * upload is waited for, as in pkv_plan_create. Returns PKV_OK and sets *out, or
 * PKV_ERR_INVALID_ARG (caps NULL, capacity below the batch) / the errors of
 * pkv_plan_create, with *out = NULL.
 */
PKV_API int pkv_plan_create_capturable(pkv_plan **out, const pkv_plan_desc *desc, const pkv_plan_caps *caps,
                                       void *stream);

/*
 * pkv_plan_update: re-plan a capturable plan for a new batch, in place: host arrays
 * in `desc` (qo_indptr, kv_indptr, kv_last_page_len, q_start, batch_size,
 * fixed_split_size, disable_split_kv) may change; kind, head counts, head_dim,
 * page_size, window_left, causal, sm_scale, dtype, kv_dtype, logits_soft_cap, k_scale,
 * v_scale, wait_limit_us, wait_probe, num_pages and the kv_indices
 * device pointer must equal the plan's (the caller rewrites that array's contents,
 * stream-ordered before the next run), else PKV_ERR_INVALID_ARG. A batch above the
 * capacity returns PKV_ERR_UNSUPPORTED and leaves the plan unchanged.
 * Allocates nothing and does not synchronise the device: the new schedule is written
 * to a pinned staging image and copied into the workspace with cudaMemcpyAsync on
 * `stream`, so runs issued later on that stream (or replays of a graph captured from
 * pkv_run) see it, and runs issued earlier see the old one. The host waits only if
 * the upload of two updates ago is still in flight. Must not be called while
 * `stream` is being captured.
 */
PKV_API int pkv_plan_update(pkv_plan *plan, const pkv_plan_desc *desc, void *stream);

/*
 * pkv_run: attention for the planned batch. q, caches and out are DEVICE bf16
 * pointers in the layouts above (16-byte aligned); lse is a DEVICE fp32 pointer or
 * NULL. All are borrowed for the duration of the launches. Asynchronous on
 * `stream`; the caller orders `stream` after whatever wrote the inputs.
 */
PKV_API int pkv_run(const pkv_plan *plan, const void *q, const void *k_cache, const void *v_cache,
            void *out, float *lse, void *stream);

/*
 * pkv_merge_state: combine two partial attention states over disjoint key sets
 * (flashinfer_backend.py, _safe_merge_state / forward_extend's ragged + paged
 * merge): for every (token, head) row,
 *     s = ln(e^s_a + e^s_b),  v = (e^s_a v_a + e^s_b v_b) / e^s,
 * where a state with s = -inf weighs nothing and two such states give v = 0,
 * s = -inf. v_*: DEVICE [n_tokens, n_heads, head_dim] of `dtype` (PKV_BF16 or
 * PKV_F32); s_*: DEVICE fp32 [n_tokens, n_heads]. v_out/s_out may alias v_a/s_a.
 * No limit on n_heads (the pages' CUDA merge fails above 1024 threads per block).
 */
PKV_API int pkv_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                    void *v_out, float *s_out, int64_t n_tokens, int32_t n_heads,
                    int32_t head_dim, int32_t dtype, void *stream);

/* Free the plan's device workspace (synchronises with nothing; do not call while
 * a run of this plan may still be executing). NULL is a no-op. */
PKV_API int pkv_plan_destroy(pkv_plan *plan);

/* Fill *info (host struct). */
PKV_API int pkv_plan_get_info(const pkv_plan *plan, pkv_plan_info *info);

/*
 * Read and clear the plan's device status word: synchronises the device, stores
 * PKV_OK or PKV_ERR_DEVICE_BOUNDS / PKV_ERR_TIMEOUT recorded by earlier runs in
 * *status, and returns PKV_OK (or PKV_ERR_CUDA if the read itself failed).
 */
PKV_API int pkv_plan_device_status(const pkv_plan *plan, int32_t *status);

/*
 * Measurement hook: record ev_begin / ev_end (cudaEvent_t passed as void*; either
 * may be NULL to stop recording it) on the run's stream immediately before and
 * after the main attention kernel of every later pkv_run of this plan, so that the
 * kernel can be timed alone (the split-KV merge pass is outside the pair).
 */
PKV_API int pkv_plan_set_timing_events(pkv_plan *plan, void *ev_begin, void *ev_end);

/*
 * pkv_decode_noalloc: the decode of pkv_plan_create + pkv_run (desc->kind must be
 * PKV_DECODE, desc->kv_dtype PKV_BF16, else PKV_ERR_UNSUPPORTED; same arguments,
 * layouts and results) in one call that allocates no
 * device memory: no cudaMalloc, cudaFree or allocating library routine. The pages
 * have no counterpart to it. It is for callers that cannot allocate: serving
 * processes whose memory pool already holds the device memory and forbids further
 * driver allocations, and latency-critical paths that cannot pay for cudaMalloc /
 * cudaFree, which may synchronise the whole device.
 *
 * The work list and the split-KV partial states live in a 32 MiB array of device
 * memory that is part of the library image: every GPU on which the library is used
 * holds it until the process exits. A batch that would need more than 32 MiB of it
 * is rejected with PKV_ERR_UNSUPPORTED before any launch (pkv_last_error() gives
 * the size; fewer splits, disable_split_kv, or pkv_plan_create + pkv_run handle it).
 * The first call on a device looks up the array's device address (with that device
 * current); make that first call before any stream capture. The work list reaches
 * the array through the arguments of small copy kernels enqueued on `stream` before
 * the decode, so the host never waits for the stream's earlier work. Every call
 * shares the array: calls whose work overlaps on the GPU (other streams, or other
 * host threads) race and must be serialised by the caller. This call has no device
 * status to read back: out-of-range page ids are skipped as in pkv_run, and a device
 * wait that gives up (PKV_ERR_TIMEOUT under pkv_run) leaves out and lse incomplete,
 * both without a report.
 */
PKV_API int pkv_decode_noalloc(const pkv_plan_desc *desc, const void *q, const void *k_cache,
                               const void *v_cache, void *out, float *lse, void *stream);

/* Static name of a status code. */
PKV_API const char *pkv_status_string(int status);

/* Reason for the last failure on the calling thread ("" if none). */
PKV_API const char *pkv_last_error(void);

/*
 * pkv_build_kv_indices: build a batch's kv_indptr and kv_indices ON THE DEVICE from a
 * request-to-slot table, so that the page table of a captured plan can be rebuilt
 * between replays without a host round trip (sglang flashinfer_backend.py page,
 * section call_begin_forward: kv_indptr is the running sum of the kept lengths, each
 * request's entries come from its table row from its start offset on, and a
 * sliding-window pool maps them into its own locations):
 *   kv_indptr[0] = 0, kv_indptr[b+1] = kv_indptr[b] + kv_lens[b]
 *   kv_indices[kv_indptr[b] + j] = req_to_token[req_pool_indices[b] * row_stride + kv_start[b] + j]
 *   then, if loc_map != NULL: kv_indices[i] = loc_map[kv_indices[i]]
 * The entries are whatever the table holds (token slots for page size 1, page ids
 * otherwise). All pointers are DEVICE int32: req_to_token [num_rows, row_stride]
 * (row-major), req_pool_indices / kv_start / kv_lens [batch_size], loc_map
 * [loc_map_len] or NULL, kv_indptr [batch_size + 1] (written), kv_indices
 * [kv_indices_capacity] (written), status: NULL or a device word in which a bounds
 * violation on the device (a row, start or map entry out of range, a negative length,
 * or more indices than kv_indices_capacity) is recorded as PKV_ERR_DEVICE_BOUNDS, the
 * offending request or entry being skipped (map misses are written as -1).
 * Asynchronous on `stream` (two kernel launches), allocates nothing; capturable.
 * Returns PKV_OK, PKV_ERR_INVALID_ARG (NULL or negative arguments) or PKV_ERR_CUDA.
 */
PKV_API int pkv_build_kv_indices(const int32_t *req_to_token, int32_t num_rows, int64_t row_stride,
                                 const int32_t *req_pool_indices, const int32_t *kv_start, const int32_t *kv_lens,
                                 int32_t batch_size, const int32_t *loc_map, int64_t loc_map_len,
                                 int32_t *kv_indptr, int32_t *kv_indices, int64_t kv_indices_capacity,
                                 int32_t *status, void *stream);

/* PKV_ABI_VERSION of the loaded library. */
PKV_API int pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
