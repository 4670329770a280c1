// Paged prefill / extend kernel on the 5th-generation tensor cores (tcgen05, TMEM),
// one 128-row query tile per CTA; used for head_dim 256 (whose two O accumulators
// would not fit TMEM next to S in the two-tile kernel).
//
// One CTA = 128 packed query rows (query tokens x the query heads that share one
// KV head, the GQA packing of flashinfer_backend.py's should_use_tensor_core) of
// one request, against the KV tiles the plan clipped to the rows' visible
// interval [p_min - W, p_max] (whole tiles outside it are never loaded: the
// tile-granular KV-start skip of sglang PR #31501, "What"). Tiles that straddle the
// window edge, the causal diagonal or the end of the cache get the exact
// per-element mask (the part the pages' bug compiled out); interior tiles skip it.
//
// Warp roles (256 threads):
//   warps 0-3  softmax + epilogue: thread r owns packed row r = TMEM lane r.
//              Reads S from TMEM, masks, keeps the fp32 running max m and sum l,
//              writes P = exp2(s - m) as bf16 into shared memory (the A operand
//              of the PV MMA), rescales O in TMEM only when m grows by more than
//              2^8 (O and l always share the same reference max, so the result is
//              exact), and finally writes out = O / l (bf16) and lse.
//   warps 4-6  producers: cp.async 16-byte gathers of Q and of each K/V tile row
//              through the page table (any page size), into 128-byte-swizzled
//              tiles; completion is signalled on mbarriers.
//   warp 7     TMEM allocation and the single MMA-issuing thread:
//              S_j = Q K_j^T (M=128, N=T, K=16 per instruction) into a
//              double-buffered TMEM S, then O += P_{j-1} V_{j-1} (M=128, N=D),
//              so S of the next tile overlaps the softmax of the current one.
// Every wait is bounded: on expiry the kernel records PKV_ERR_TIMEOUT, releases
// the other roles through a shared abort flag, drains its MMAs, frees TMEM and
// returns.
#include <cfloat>
#include <climits>

#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
namespace {

template <int D>
struct PrefillTraits {
    static constexpr int kM = kPrefillRows;            // packed query rows per CTA
    static constexpr int kT = D >= 256 ? 64 : 128;     // KV tokens per tile
    static constexpr int kStages = 2;
    static constexpr int kChunk = 128;                 // bytes per swizzled row (64 bf16)
    static constexpr int kQBytes = kM * D * 2;
    static constexpr int kKVBytes = kT * D * 2;
    static constexpr int kPBytes = kM * kT * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kDynSmem = kOffP + kPBytes + 1024;  // + alignment slack
    static constexpr int kTmemCols = 512;
    static constexpr int kTmemO = 256;                 // O columns; S buffer b at b * kT
    static constexpr int kThreads = 256;
    static constexpr int kProducers = 96;              // producer threads (warps 4-6)
    static_assert(2 * kT <= kTmemO && kTmemO + D <= kTmemCols, "TMEM budget");
};

constexpr long long kWaitLimit = 4000000000LL;  // clock cycles (about 2 s)

// Barrier slots.
template <int S>
struct Bars {
    static constexpr int kQ = 0;
    static constexpr int kKFull = 1;
    static constexpr int kVFull = kKFull + S;
    static constexpr int kKVEmpty = kVFull + S;
    static constexpr int kSFull = kKVEmpty + S;  // 2
    static constexpr int kPFull = kSFull + 2;
    static constexpr int kPVDone = kPFull + 1;
    static constexpr int kDrain = kPVDone + 1;
    static constexpr int kCount = kDrain + 1;
};

template <int D, int MASK>
__global__ void __launch_bounds__(256, 1) prefill_kernel(const PrefillParams p)
{
    using Tr = PrefillTraits<D>;
    using B = Bars<Tr::kStages>;
    constexpr int T = Tr::kT;
    constexpr int S = Tr::kStages;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    constexpr bool kCausal = MASK == kMaskCausal || MASK == kMaskCausalWindow;
    constexpr bool kWindow = MASK == kMaskCausalWindow || MASK == kMaskWindow;

    extern __shared__ uint8_t dsmem_raw[];
    __shared__ __align__(8) uint64_t bars[B::kCount];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    __shared__ int no_abort;

    const uint32_t base = (smem_u32(dsmem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base + Tr::kOffQ;
    const uint32_t sK = base + Tr::kOffK;
    const uint32_t sV = base + Tr::kOffV;
    const uint32_t sP = base + Tr::kOffP;
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const PrefillItem it = p.items[blockIdx.x];
    const RequestInfo rq = p.reqs[it.req];
    const int n_tiles = it.kv_tile_hi - it.kv_tile_lo;
    const int g = p.group;
    const int valid_rows = it.ntok * g;
    const volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        mbar_init(bar(B::kQ), Tr::kProducers);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(B::kKFull + s), Tr::kProducers);
            mbar_init(bar(B::kVFull + s), Tr::kProducers);
            mbar_init(bar(B::kKVEmpty + s), 1);
        }
        mbar_init(bar(B::kSFull + 0), 1);
        mbar_init(bar(B::kSFull + 1), 1);
        mbar_init(bar(B::kPFull), 128);
        mbar_init(bar(B::kPVDone), 1);
        mbar_init(bar(B::kDrain), 1);
        abort_flag = 0;
        no_abort = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 7) {
        tmem_alloc(smem_u32(&tmem_base_s), Tr::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp < 4) {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x;
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        const int tok = it.tok0 + r / g;
        const int pos = rq.q_start + tok;
        const int p_min = rq.q_start + it.tok0;
        const int p_max = p_min + it.ntok - 1;
        const float scale = p.sm_scale_log2;
        float m_used = -INFINITY;
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int buf = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull + buf), (j >> 1) & 1, abort_v, kWaitLimit));
            if (!ok)
                break;
            tc_fence_after();
            float s[T];
#pragma unroll
            for (int c = 0; c < T / 32; ++c)
                tmem_ld32(t_lane + buf * T + 32 * c, *reinterpret_cast<float(*)[32]>(&s[32 * c]));
            tmem_wait_ld();

            const int j0 = (it.kv_tile_lo + j) * T;
            bool need_mask = j0 + T > rq.kv_len;
            if (kCausal)
                need_mask |= j0 + T - 1 > p_min;
            if (kWindow)
                need_mask |= j0 < p_max - p.window_left;
            if (need_mask) {
                const int lo_c = kWindow ? pos - p.window_left - j0 : INT_MIN;
                int hi_c = rq.kv_len - 1 - j0;
                if (kCausal)
                    hi_c = min(hi_c, pos - j0);
#pragma unroll
                for (int c = 0; c < T; ++c)
                    s[c] = (c >= lo_c && c <= hi_c) ? s[c] * scale : -INFINITY;
            } else {
#pragma unroll
                for (int c = 0; c < T; ++c)
                    s[c] *= scale;
            }
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mx8[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
            for (int c = 16; c < T; c += 8)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mx8[k] = fmaxf(mx8[k], s[c + k]);
            const float m_tile = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_cand = fmaxf(m_used, m_tile);
            const bool need = m_cand != -INFINITY && (m_used == -INFINITY || m_cand > m_used + 8.f);
            const float alpha = need ? fast_exp2(m_used - m_cand) : 1.f;

            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kPVDone), (j - 1) & 1, abort_v, kWaitLimit));
                if (!ok)
                    break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(t_lane + Tr::kTmemO + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] *= alpha;
                        tmem_st32(t_lane + Tr::kTmemO + 32 * c, o);
                    }
                    tmem_wait_st();
                }
            }
            if (need) {
                l *= alpha;
                m_used = m_cand;
            }
            const float ref = m_used == -INFINITY ? 0.f : m_used;
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c8 = 0; c8 < T / 8; ++c8) {
                float e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    e[k] = fast_exp2(s[8 * c8 + k] - ref);
                    rs[k & 3] += e[k];
                }
                const uint32_t w0 = pack_bf16(e[0], e[1]), w1 = pack_bf16(e[2], e[3]);
                const uint32_t w2 = pack_bf16(e[4], e[5]), w3 = pack_bf16(e[6], e[7]);
                const uint32_t dst = sP + (c8 >> 3) * (Tr::kM * Tr::kChunk) + r * Tr::kChunk +
                                     (((c8 & 7) ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst), "r"(w0), "r"(w1),
                             "r"(w2), "r"(w3)
                             : "memory");
            }
            l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B::kPFull));
        }
        if (ok && n_tiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kPVDone), (n_tiles - 1) & 1, abort_v, kWaitLimit));
            tc_fence_after();
        }
        if (!ok) {
            record_status(p.status, PKV_ERR_TIMEOUT);
            abort_flag = 1;
        } else {
            const bool row_ok = r < valid_rows;
            const int h = it.kv_head * g + r % g;
            const size_t orow = ((size_t)(rq.qo_begin + tok) * p.num_qo_heads + h);
            uint16_t *dst = p.out + orow * D;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                if (n_tiles > 0) {
                    tmem_ld32(t_lane + Tr::kTmemO + 32 * c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = 0.f;
                }
                if (row_ok) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack_bf16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                        v.y = pack_bf16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                        v.z = pack_bf16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                        v.w = pack_bf16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                        *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * q4) = v;
                    }
                }
            }
            if (row_ok && p.lse)
                p.lse[orow] = l > 0.f ? (m_used + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
    } else if (warp < 7) {
        // ------------------------------------------------------------ producers
        constexpr int NP = Tr::kProducers;
        const int pt = threadIdx.x - 128;
        for (int idx = pt; idx < Tr::kM * CH; idx += NP) {
            const int r = idx / CH, c = idx % CH;
            const bool v = r < valid_rows;
            const int rr = v ? r : 0;
            const uint16_t *src = p.q + ((size_t)(rq.qo_begin + it.tok0 + rr / g) * p.num_qo_heads +
                                         it.kv_head * g + rr % g) * D + c * 8;
            const uint32_t dst = sQ + (c >> 3) * (Tr::kM * Tr::kChunk) + r * Tr::kChunk + (((c & 7) ^ (r & 7)) << 4);
            cp_async_16(dst, src, v ? 16u : 0u);
        }
        cp_async_mbar_arrive(bar(B::kQ));

        constexpr int kPerThread = (T * CH + NP - 1) / NP;  // 16-byte chunks per thread per tile
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % S;
            if (j >= S) {
                if (!mbar_wait(bar(B::kKVEmpty + st), ((j / S) + 1) & 1, abort_v, kWaitLimit)) {
                    record_status(p.status, PKV_ERR_TIMEOUT);
                    abort_flag = 1;
                    break;
                }
            }
            const int j0 = (it.kv_tile_lo + j) * T;
            size_t off[kPerThread];
            uint32_t bytes[kPerThread];
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const int idx = pt + NP * k;
                const int t = idx / CH, c = idx % CH;
                const int jj = j0 + t;
                off[k] = 0;
                bytes[k] = 0;
                if (idx < T * CH && jj < rq.kv_len) {
                    const int lp = p.page_shift >= 0 ? (jj >> p.page_shift) : jj / p.page_size;
                    const int slot = jj - lp * p.page_size;
                    const int page = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                    if ((unsigned)page < (unsigned)p.num_pages) {
                        off[k] = (((size_t)page * p.page_size + slot) * p.num_kv_heads + it.kv_head) * D + c * 8;
                        bytes[k] = 16;
                    } else {
                        record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                    }
                }
            }
            const uint32_t kbase = sK + st * Tr::kKVBytes;
            const uint32_t vbase = sV + st * Tr::kKVBytes;
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const int idx = pt + NP * k;
                const int t = idx / CH, c = idx % CH;
                const uint32_t so = (c >> 3) * (T * Tr::kChunk) + t * Tr::kChunk + (((c & 7) ^ (t & 7)) << 4);
                if (idx < T * CH)
                    cp_async_16(kbase + so, p.k_cache + off[k], bytes[k]);
            }
            cp_async_mbar_arrive(bar(B::kKFull + st));
#pragma unroll
            for (int k = 0; k < kPerThread; ++k) {
                const int idx = pt + NP * k;
                const int t = idx / CH, c = idx % CH;
                const uint32_t so = (c >> 3) * (T * Tr::kChunk) + t * Tr::kChunk + (((c & 7) ^ (t & 7)) << 4);
                if (idx < T * CH)
                    cp_async_16(vbase + so, p.v_cache + off[k], bytes[k]);
            }
            cp_async_mbar_arrive(bar(B::kVFull + st));
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(Tr::kM, T, false);
            const uint32_t idesc_o = idesc_bf16_f32(Tr::kM, D, true);
            bool ok = n_tiles == 0 || mbar_wait(bar(B::kQ), 0, abort_v, kWaitLimit);
            for (int j = 0; ok && j <= n_tiles && n_tiles > 0; ++j) {
                if (j < n_tiles) {
                    const int st = j % S, buf = j & 1;
                    ok = mbar_wait(bar(B::kKFull + st), (j / S) & 1, abort_v, kWaitLimit);
                    if (!ok)
                        break;
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t kb = sK + st * Tr::kKVBytes;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t a = sdesc_sw128(sQ + (k >> 2) * (Tr::kM * Tr::kChunk) + (k & 3) * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(kb + (k >> 2) * (T * Tr::kChunk) + (k & 3) * 32, 16, 1024);
                        umma_f16(tmem + buf * T, a, b, idesc_s, k > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(B::kSFull + buf));
                }
                if (j >= 1) {
                    const int i = j - 1, st = i % S;
                    ok = mbar_wait(bar(B::kPFull), i & 1, abort_v, kWaitLimit) &&
                         mbar_wait(bar(B::kVFull + st), (i / S) & 1, abort_v, kWaitLimit);
                    if (!ok)
                        break;
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t vb = sV + st * Tr::kKVBytes;
#pragma unroll
                    for (int k = 0; k < T / 16; ++k) {
                        const uint64_t a = sdesc_sw128(sP + (k >> 2) * (Tr::kM * Tr::kChunk) + (k & 3) * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(vb + k * (16 * Tr::kChunk), T * Tr::kChunk, 1024);
                        umma_f16(tmem + Tr::kTmemO, a, b, idesc_o, (i > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(B::kPVDone));
                    umma_commit(bar(B::kKVEmpty + st));
                }
            }
            if (!ok) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
            }
            // Every MMA issued above has completed once this barrier flips.
            umma_commit(bar(B::kDrain));
            mbar_wait(bar(B::kDrain), 0, &no_abort, kWaitLimit);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 7) {
        tc_fence_after();
        tmem_dealloc(tmem, Tr::kTmemCols);
    }
}

template <int D, int MASK>
cudaError_t launch_prefill_dm(const PrefillParams &p, int num_items, cudaStream_t s)
{
    using Tr = PrefillTraits<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, MASK>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kDynSmem);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    prefill_kernel<D, MASK><<<num_items, Tr::kThreads, Tr::kDynSmem, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_d(const PrefillParams &p, int mask_mode, int num_items, cudaStream_t s)
{
    switch (mask_mode) {
    case kMaskNone: return launch_prefill_dm<D, kMaskNone>(p, num_items, s);
    case kMaskCausal: return launch_prefill_dm<D, kMaskCausal>(p, num_items, s);
    case kMaskCausalWindow: return launch_prefill_dm<D, kMaskCausalWindow>(p, num_items, s);
    case kMaskWindow: return launch_prefill_dm<D, kMaskWindow>(p, num_items, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int prefill_kv_tile(int head_dim) { return head_dim >= 256 ? 64 : 128; }

cudaError_t launch_prefill(const PrefillParams &p, int head_dim, int mask_mode, int num_items, cudaStream_t s)
{
    // head_dim 64 and 128 run the two-tile kernel of pkv_prefill_pp.cu.
    return head_dim == 256 ? launch_prefill_d<256>(p, mask_mode, num_items, s) : cudaErrorInvalidValue;
}

}  // namespace pkv
