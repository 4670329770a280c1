// Split-KV paged decode kernel: one query row per request, the whole query-head
// group of a KV head against each streamed K/V row (GQA packing: the query-head group
// forms the MMA rows, as the sglang flashinfer_backend.py page, section
// should_use_tensor_core, describes for its tensor-core decode), online softmax
// in fp32, fp32 partial states per split for the merge pass.
//
// The plan has already clipped each CTA's key range [j0, j1) to the visible
// interval [p - W, p] of the request's single query position, so every key inside
// the range is visible; the kernel masks only what lies outside it in the first
// and last stage.
//
// CTA = TT/TPW compute warps + 1 producer warp. bf16 caches: TT = 64 tokens per stage
// (160 threads, 2 CTAs per SM) or, for batches of short key ranges, 32 (96 threads,
// 4 CTAs per SM), TPW = 16 tokens per compute warp. 8-bit caches (E4M3 / E5M2): the
// same two CTA shapes with stages of 128 and 64 tokens, TPW = 32 (two independent
// 16-token sub-blocks per warp), K and V widened to f16 in registers before the MMAs.
//   producer: fills a ring of shared-memory stages (TT tokens of K and of V each,
//     stored as 128-byte-swizzled planes) either with TMA boxes of whole pages (a
//     4-D tensor map over [page, slot, KV head, d]; the page ids of the next tile
//     are fetched while the current one is issued) when the page size is a multiple
//     of 8 that divides TT or is a multiple of it, or else with 16-byte cp.async
//     gathers; completion through mbarriers;
//   compute warp w: tokens [TPW w, TPW w + TPW) of every stage, S = Q K^T and
//     O += P V with mma.sync m16n8k16 (bf16, or f16 for 8-bit caches, in; fp32
//     accumulate; rows = the query heads), running its own (m, l, O) without
//     CTA-wide barriers; the warps' states are merged once at the end. A CTA that
//     handles one split of a request writes an fp32 partial state; the group's
//     last CTA to finish (an arrival counter after a memory fence) combines the
//     partials through their LSE, so no second kernel runs.
// All waits are bounded (the plan's wait bound, 2 s by default); on expiry
// PKV_ERR_TIMEOUT is recorded and the CTA winds down after its outstanding copies
// have landed.
#pragma once

#include <cfloat>

#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
namespace dec {

// TT = KV tokens per stage: 64 (the general kernel, 2 CTAs per SM at d <= 128) or
// 32 for batches of short key ranges (two compute warps and a 48 KB ring at d 128,
// 4 CTAs per SM, so that a batch of short ranges runs in one wave).
// KV = element type of the caches: PKV_BF16, PKV_FP8_E4M3 or PKV_FP8_E5M2. An 8-bit
// tile takes half the bytes, so the ring holds twice the stages (the same bytes in
// flight per SM).
template <int D, int TT, int KV = PKV_BF16, int TPW = 16>
struct DecTraits {
    static constexpr int kElem = KV == PKV_BF16 ? 2 : 1;  // bytes per cache element
    static constexpr int kRowBytes = D * kElem;            // one token of one head
    static constexpr int kPlaneRow = kRowBytes < 128 ? kRowBytes : 128;  // bytes per row of a plane
    static constexpr int kTile = TT;
    static constexpr int kCompute = TT / TPW;  // compute warps, TPW tokens of each tile apiece
    static constexpr int kThreads = 32 * (kCompute + 1);  // + one producer warp
    static constexpr int kNCh = kRowBytes / kPlaneRow;    // swizzled column planes
    static constexpr int kGran = kRowBytes / 16;          // 16-byte granules per row
    static constexpr int kPlaneBytes = kTile * kPlaneRow;
    static constexpr int kTileBytes = kTile * kRowBytes;  // K or V of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    // Stages: about the same bytes in flight per SM for every variant.
    static constexpr int kStages =
        (TT == 128 || (TT == 64 && TPW == 32)) ? 3 : (D == 64 ? 4 : 3) * (kElem == 1 ? 2 : 1);
    static constexpr int kORowFloats = D + 8;  // padded row of the combine buffer
    static constexpr int kCombineBytes = kCompute * kDecodeRows * kORowFloats * 4;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kDynSmem = (kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes) + 1024;
    // two compute warps (96 threads): 4 CTAs per SM, so a batch of short ranges runs in one wave
    static constexpr int kMinBlocks = kCompute == 2 ? 4 : (D >= 256 ? 1 : 2);
};

// Byte offset of 16-byte granule `c16` of row `row` in a TT-row tile stored as
// planes of PR-byte rows: PR = 128 with the 128-byte XOR swizzle (the layout a
// SWIZZLE_128B TMA box produces; granules 8 apart sit in the next plane), or PR = 64
// (one 64-byte row per token, 8-bit d 64) with the 64-byte swizzle of SWIZZLE_64B.
// GM > 0 (bf16 caches, GM = 128-byte planes per row): group-major, 8-row groups of all
// GM planes [TT/8][GM][8 rows][128 B], so that one TMA box of a page brings every
// plane of its rows; otherwise plane-major [planes][TT rows][PR bytes].
template <int TT, int PR = 128, int GM = 0>
__device__ __forceinline__ uint32_t plane_off(int row, int c16)
{
    if (PR == 64)
        return (uint32_t)(row * 64 + (((c16 & 3) ^ ((row >> 1) & 3)) << 4));
    if (GM > 0)
        return (uint32_t)((row >> 3) * (GM * 1024) + (c16 >> 3) * 1024 + (row & 7) * 128 +
                          (((c16 & 7) ^ (row & 7)) << 4));
    return (uint32_t)((c16 >> 3) * (TT * 128) + row * 128 + (((c16 & 7) ^ (row & 7)) << 4));
}

// Four 8-bit values (a 32-bit word, lowest byte first) as two f16x2 words: {x0, x1}
// and {x2, x3}. Every E4M3 and E5M2 value is exact in f16; an E5M2 byte is the top
// byte of its f16, so that format needs only byte moves.
template <int KV>
__device__ __forceinline__ void fp8x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    if (KV == PKV_FP8_E5M2) {
        lo = __byte_perm(w, 0u, 0x1404);
        hi = __byte_perm(w, 0u, 0x3424);
    } else {
        asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
            " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    }
}

// The same for a word of a transposed V load, whose bytes are (token 2c, column 2n),
// (2c, 2n+1), (2c+1, 2n), (2c+1, 2n+1): even = f16x2 of column 2n for tokens 2c, 2c+1,
// odd = the same for column 2n+1.
template <int KV>
__device__ __forceinline__ void fp8x4_pairs_to_f16x2(uint32_t w, uint32_t &even, uint32_t &odd)
{
    if (KV == PKV_FP8_E5M2) {
        even = __byte_perm(w, 0u, 0x2404);
        odd = __byte_perm(w, 0u, 0x3414);
    } else {
        fp8x4_to_f16x2<KV>(__byte_perm(w, 0u, 0x3120), even, odd);
    }
}

template <int D, bool TMA_KV, int TT, int KV, int TPW>
__global__ void __launch_bounds__(DecTraits<D, TT, KV, TPW>::kThreads, DecTraits<D, TT, KV, TPW>::kMinBlocks)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v)
{
    using Tr = DecTraits<D, TT, KV, TPW>;
    constexpr int NSB = TPW / 16;  // 16-token sub-blocks per compute warp
    constexpr bool KV8 = KV != PKV_BF16;
    constexpr int PR = Tr::kPlaneRow;
    constexpr int GM = KV8 ? 0 : Tr::kNCh;  // bf16: group-major stages (one TMA box per page)
    constexpr int S = Tr::kStages;
    constexpr int NW = Tr::kCompute;
    constexpr int NT = 32 * NW;  // compute threads
    extern __shared__ uint8_t dsmem_raw[];
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ float red_m[NW][kDecodeRows];
    __shared__ float red_l[NW][kDecodeRows];
    __shared__ float row_m[kDecodeRows];
    __shared__ float row_inv_l[kDecodeRows];
    __shared__ __align__(8) uint64_t never_bar;  // the wait probe's barrier: nothing completes it
    __shared__ int abort_flag;
    __shared__ int no_abort;

    const uint32_t ring = (smem_u32(dsmem_raw) + 1023u) & ~1023u;
    uint8_t *ring_gen = dsmem_raw + (ring - smem_u32(dsmem_raw));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (p.live_items && (int)blockIdx.x >= *p.live_items)
        return;  // a capturable plan's fixed grid: this CTA has no work item now
    const DecodeItem it = p.items[blockIdx.x];
    struct {
        int32_t qo_begin, kv_len, kv_page_begin;
    } const rq = {it.row, it.kv_len, it.kv_page_begin};
    const int tb = it.j1 > it.j0 ? (it.j0 / TT) * TT : it.j0;  // first tile start (64-aligned)
    const int ntiles = it.j1 > it.j0 ? (it.j1 - tb + TT - 1) / TT : 0;
    const volatile int *abort_v = &abort_flag;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), TMA_KV ? 1 : 32);
            mbar_init(smem_u32(&empty_bar[s]), Tr::kCompute);
        }
        mbar_init(smem_u32(&never_bar), 1);
        abort_flag = 0;
        no_abort = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    // Everything above reads only the plan's own data; q, the caches and the page
    // table may come from the previous kernel in the stream.
    grid_dependency_wait();

    if (warp == Tr::kCompute) {
        // ------------------------------------------------------------ producer
        const int P = p.page_size;
        int issued = 0;
        bool ok = true;
        if (TMA_KV) {
            const int rows_box = P < TT ? P : TT;
            const int npg = TT / rows_box;
            const int n_pages_req = (rq.kv_len + P - 1) / P;
            auto load_id = [&](int t) -> int {
                if (lane >= npg)
                    return -1;
                const int ts = tb + t * TT;
                const int lp = P <= TT ? ts / P + lane : ts / P;
                const int first = P <= TT ? lp * P : ts;
                // pages holding no key of [j0, j1) are not loaded
                if (lp >= n_pages_req || first >= it.j1 || first + rows_box <= it.j0)
                    return -1;
                const int pg = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                if ((unsigned)pg >= (unsigned)p.num_pages) {
                    record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                    return -1;
                }
                return pg;
            };
            if (lane == 0) {
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            int pg = ntiles > 0 ? load_id(0) : -1;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % S;
                const int pg_next = t + 1 < ntiles ? load_id(t + 1) : -1;
                if (t >= S) {
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[s]), ((t / S) - 1) & 1, abort_v,
                                                          p.wait_ns));
                    if (!ok)
                        break;
                }
                const int ts = tb + t * TT;
                const int slot0 = P > TT ? ts % P : 0;
                const unsigned valid = __ballot_sync(0xffffffffu, pg >= 0);
                if (lane == 0)
                    mbar_arrive_expect_tx(smem_u32(&full_bar[s]),
                                          (uint32_t)__popc(valid) * rows_box * PR * Tr::kNCh * 2);
                __syncwarp();
                if (pg >= 0) {
                    const uint32_t kb = ring + s * Tr::kStageBytes;
                    const uint32_t vb = kb + Tr::kTileBytes;
                    if (GM > 0) {
                        // one 5-D box [8-row blocks][H_kv][plane][8 rows][64] per page: all planes
                        const uint32_t o = (uint32_t)(lane * rows_box / 8) * (GM * 1024);
                        const int blk = (pg * P + slot0) >> 3;
                        tma_load_5d(kb + o, &tm_k, 0, 0, 0, it.kv_head, blk, smem_u32(&full_bar[s]));
                        tma_load_5d(vb + o, &tm_v, 0, 0, 0, it.kv_head, blk, smem_u32(&full_bar[s]));
                    } else {
                        for (int c = 0; c < Tr::kNCh; ++c) {
                            const uint32_t o = c * Tr::kPlaneBytes + lane * rows_box * PR;
                            const int x = c * (PR / Tr::kElem);  // first element of the plane
                            tma_load_4d(kb + o, &tm_k, x, it.kv_head, slot0, pg, smem_u32(&full_bar[s]));
                            tma_load_4d(vb + o, &tm_v, x, it.kv_head, slot0, pg, smem_u32(&full_bar[s]));
                        }
                    }
                }
                issued = t + 1;
                pg = pg_next;
            }
        } else {
            constexpr int CH = Tr::kGran;
            const uint8_t *kcache = reinterpret_cast<const uint8_t *>(p.k_cache);
            const uint8_t *vcache = reinterpret_cast<const uint8_t *>(p.v_cache);
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % S;
                if (t >= S) {
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[s]), ((t / S) - 1) & 1, abort_v,
                                                          p.wait_ns));
                    if (!ok)
                        break;
                }
                const int ts = tb + t * TT;
                const uint32_t kb = ring + s * Tr::kStageBytes;
                const uint32_t vb = kb + Tr::kTileBytes;
#pragma unroll
                for (int rr = 0; rr < TT / 32; ++rr) {
                    const int row = lane + 32 * rr;
                    const int j = ts + row;
                    size_t off = 0;
                    uint32_t bytes = 0;
                    if (j >= it.j0 && j < it.j1) {
                        const int lp = p.page_shift >= 0 ? (j >> p.page_shift) : j / P;
                        const int page = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                        if ((unsigned)page < (unsigned)p.num_pages) {
                            off = (((size_t)page * P + (j - lp * P)) * p.num_kv_heads + it.kv_head) *
                                  Tr::kRowBytes;
                            bytes = 16;
                        } else {
                            record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < CH; ++c) {
                        cp_async_16(kb + plane_off<TT, PR, GM>(row, c), kcache + off + c * 16, bytes);
                        cp_async_16(vb + plane_off<TT, PR, GM>(row, c), vcache + off + c * 16, bytes);
                    }
                }
                cp_async_mbar_arrive(smem_u32(&full_bar[s]));
                issued = t + 1;
            }
        }
        if (!ok && lane == 0) {
            record_status(p.status, PKV_ERR_TIMEOUT);
            abort_flag = 1;
        }
        // Never leave with copies in flight: wait for the last stages issued.
        for (int t = issued - S < 0 ? 0 : issued - S; t < issued; ++t)
            mbar_wait(smem_u32(&full_bar[t % S]), (t / S) & 1, &no_abort, p.wait_ns);
        if (!TMA_KV)
            asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else {
        // ------------------------------------------------------------ compute
        // Q fragments straight from global memory (rows >= nheads are zero).
        uint32_t qf[D / 16][4];
        {
            const int r0 = lane >> 2, r1 = r0 + 8;
            const uint32_t *q0 = reinterpret_cast<const uint32_t *>(
                p.q + ((size_t)rq.qo_begin * p.num_qo_heads + it.head0 + (r0 < it.nheads ? r0 : 0)) * D);
            const uint32_t *q1 = reinterpret_cast<const uint32_t *>(
                p.q + ((size_t)rq.qo_begin * p.num_qo_heads + it.head0 + (r1 < it.nheads ? r1 : 0)) * D);
            const bool v0 = r0 < it.nheads, v1 = r1 < it.nheads;
            if (!KV8) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks * 8 + (lane & 3);  // 32-bit word: columns 2c, 2c+1
                    qf[ks][0] = v0 ? __ldg(q0 + c) : 0u;
                    qf[ks][1] = v1 ? __ldg(q1 + c) : 0u;
                    qf[ks][2] = v0 ? __ldg(q0 + c + 4) : 0u;
                    qf[ks][3] = v1 ? __ldg(q1 + c + 4) : 0u;
                }
            } else {
                // 8-bit K: the k-slots of k-step ks take the columns 16ks + 4c .. 16ks + 4c + 3
                // (c = lane & 3) in the order a 32-bit ldmatrix word of the 8-bit K tile
                // holds them (slots 2c, 2c+1 <- columns 4c, 4c+1; slots 2c+8, 2c+9 <- 4c+2,
                // 4c+3): the dot product does not depend on the order of its terms.
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int c = ks * 8 + 2 * (lane & 3);
                    qf[ks][0] = v0 ? __ldg(q0 + c) : 0u;
                    qf[ks][1] = v1 ? __ldg(q1 + c) : 0u;
                    qf[ks][2] = v0 ? __ldg(q0 + c + 1) : 0u;
                    qf[ks][3] = v1 ? __ldg(q1 + c + 1) : 0u;
                }
            }
        }
        // 8-bit K runs f16 MMAs (E4M3 and E5M2 are exact in f16; bf16 is not): q is
        // scaled by 2^qe, qe chosen so that max |q| * 2^qe lies in [2^13, 2^14), and
        // rounded to f16 (exact for every entry above 2^-28 max |q|); the logits are
        // scaled back by 2^-qe.
        float q_unscale = 1.f;
        if (KV8) {
            float amax = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    amax = max3f(amax, fabsf(__uint_as_float(qf[ks][r] << 16)),
                                 fabsf(__uint_as_float(qf[ks][r] & 0xffff0000u)));
#pragma unroll
            for (int sh = 16; sh >= 1; sh >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
            int qe = 13 - ((int)((__float_as_uint(amax) >> 23) & 0xff) - 127);
            qe = qe < -100 ? -100 : (qe > 100 ? 100 : qe);
            const float up = __uint_as_float((uint32_t)(127 + qe) << 23);
            q_unscale = __uint_as_float((uint32_t)(127 - qe) << 23);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    qf[ks][r] = pack_f16(__uint_as_float(qf[ks][r] << 16) * up,
                                         __uint_as_float(qf[ks][r] & 0xffff0000u) * up);
        }
        float m[2] = {-INFINITY, -INFINITY};
        float l[2] = {0.f, 0.f};
        float o[D / 8][4];
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        const float scale = p.sm_scale_log2 * q_unscale;  // raw MMA dot -> log2-domain logit
        const float cap_in = p.cap_in * q_unscale;         // raw MMA dot -> tanh argument
        const float cap_scale = p.cap_out * p.sm_scale_log2;  // tanh -> log2-domain logit
        bool ok = true;

        for (int t = 0; t < ntiles; ++t) {
            const int s = t % S;
            // (the wait probe replaces the first stage's barrier by one nothing completes)
            const uint32_t fb = (p.wait_probe && t == 0) ? smem_u32(&never_bar) : smem_u32(&full_bar[s]);
            ok = __all_sync(0xffffffffu, mbar_wait(fb, (t / S) & 1, abort_v, p.wait_ns));
            if (!ok)
                break;
            const uint32_t kb = ring + s * Tr::kStageBytes;
            const uint32_t vb = kb + Tr::kTileBytes;
            const int wt0 = tb + t * TT + warp * TPW;  // first token of this warp's TPW
            const bool partial = wt0 < it.j0 || wt0 + TPW > it.j1;
            if (TMA_KV && partial) {
                // V rows outside [j0, j1) hold other keys, foreign slots or stale
                // data: zero them so that P = 0 never meets a non-finite value.
                uint8_t *vgen = ring_gen + s * Tr::kStageBytes + Tr::kTileBytes;
                for (int e = lane; e < TPW * Tr::kGran; e += 32) {
                    const int row = warp * TPW + e / Tr::kGran, c = e % Tr::kGran;
                    const int j = tb + t * TT + row;
                    if (j < it.j0 || j >= it.j1)
                        *reinterpret_cast<uint4 *>(vgen + plane_off<TT, PR, GM>(row, c)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // S for each 16-token sub-block b of the warp: even and odd k-steps
            // accumulate apart (sc, sc2) and are added at the end, which halves the
            // dependent MMA chain; the sub-blocks are independent chains.
            float sc[NSB][2][4], sc2[NSB][2][4];
#pragma unroll
            for (int b = 0; b < NSB; ++b)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sc[b][nt][e] = sc2[b][nt][e] = 0.f;
#pragma unroll
            for (int b = 0; b < NSB; ++b) {
                const int row0 = warp * TPW + 16 * b;
                if (!KV8) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int mi = lane >> 3;
                        const int row = row0 + ((mi >> 1) << 3) + (lane & 7);
                        const int c16 = 2 * ks + (mi & 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kb + plane_off<TT, 128, GM>(row, c16), b0, b1, b2, b3);
                        float (&acc)[2][4] = (ks & 1) ? sc2[b] : sc[b];
                        mma_bf16_16816(acc[0], qf[ks], b0, b1);
                        mma_bf16_16816(acc[1], qf[ks], b2, b3);
                    }
                } else {
                    // One 16-byte granule of an 8-bit K row = the 16 columns of one
                    // k-step. Matrix m of the x4 load: tokens 8(m & 1) .. +7, granule
                    // 2kk + (m >> 1); each word holds token lane/4's columns 4c .. 4c+3.
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const int mi = lane >> 3;
                        const int row = row0 + ((mi & 1) << 3) + (lane & 7);
                        uint32_t w[4];
                        ldmatrix_x4(kb + plane_off<TT, PR, GM>(row, 2 * kk + (mi >> 1)), w[0], w[1], w[2], w[3]);
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            uint32_t b0, b1;
                            fp8x4_to_f16x2<KV>(w[m], b0, b1);
                            mma_f16_16816((m >> 1) ? sc2[b][m & 1] : sc[b][m & 1], qf[2 * kk + (m >> 1)], b0, b1);
                        }
                    }
                }
            }
            // log2-domain logits: the soft cap on the scaled dot product, or the plain
            // scaled dot (a uniform branch); then the mask, on the edge tiles only.
            if (p.cap_in > 0.f) {
#pragma unroll
                for (int b = 0; b < NSB; ++b)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[b][nt][e] = cap_scale * soft_cap_tanh((sc[b][nt][e] + sc2[b][nt][e]) * cap_in);
            } else {
#pragma unroll
                for (int b = 0; b < NSB; ++b)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[b][nt][e] = (sc[b][nt][e] + sc2[b][nt][e]) * scale;
            }
            if (partial) {
#pragma unroll
                for (int b = 0; b < NSB; ++b) {
                    const int tok_base = wt0 + 16 * b + 2 * (lane & 3);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = tok_base + nt * 8 + (e & 1);
                            if (j < it.j0 || j >= it.j1)
                                sc[b][nt][e] = -INFINITY;
                        }
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int b = 0; b < NSB; ++b) {
                mx0 = fmaxf(mx0, fmaxf(fmaxf(sc[b][0][0], sc[b][0][1]), fmaxf(sc[b][1][0], sc[b][1][1])));
                mx1 = fmaxf(mx1, fmaxf(fmaxf(sc[b][0][2], sc[b][0][3]), fmaxf(sc[b][1][2], sc[b][1][3])));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
            const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
            const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = fast_exp2(m[0] - ref0), a1 = fast_exp2(m[1] - ref1);
            m[0] = mn0;
            m[1] = mn1;
            // P = 2^(s - m) overwrites the scores
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int b = 0; b < NSB; ++b)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    sc[b][nt][0] = fast_exp2(sc[b][nt][0] - ref0);
                    sc[b][nt][1] = fast_exp2(sc[b][nt][1] - ref0);
                    sc[b][nt][2] = fast_exp2(sc[b][nt][2] - ref1);
                    sc[b][nt][3] = fast_exp2(sc[b][nt][3] - ref1);
                    ls0 += sc[b][nt][0] + sc[b][nt][1];
                    ls1 += sc[b][nt][2] + sc[b][nt][3];
                }
            l[0] = l[0] * a0 + ls0;
            l[1] = l[1] * a1 + ls1;
            // O is rescaled only when a row maximum of the warp moved (a = 1 otherwise:
            // skipping the multiply changes nothing).
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    o[i][0] *= a0;
                    o[i][1] *= a0;
                    o[i][2] *= a1;
                    o[i][3] *= a1;
                }
            }
#pragma unroll
            for (int b = 0; b < NSB; ++b) {
                const int row0 = warp * TPW + 16 * b;
                const float (&pr)[2][4] = sc[b];
                if (!KV8) {
                    const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                                            pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
#pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        const int mi = lane >> 3;
                        const int row = row0 + ((mi & 1) << 3) + (lane & 7);
                        const int c16 = 2 * np + (mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(vb + plane_off<TT, 128, GM>(row, c16), b0, b1, b2, b3);
                        mma_bf16_16816(o[2 * np], pa, b0, b1);
                        mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
                    }
                } else {
                    // P in f16 (values in [0, 1]). A transposed x4 load of the 8-bit V
                    // tile gives, per word, tokens 2c and 2c+1 (c = lane & 3) of columns
                    // 2n, 2n+1 (n = lane / 4) of one granule; a byte permute pairs the two
                    // tokens of each column. o[2g] then accumulates the even columns
                    // 16g + 2n of granule g, o[2g + 1] the odd ones.
                    const uint32_t pa[4] = {pack_f16(pr[0][0], pr[0][1]), pack_f16(pr[0][2], pr[0][3]),
                                            pack_f16(pr[1][0], pr[1][1]), pack_f16(pr[1][2], pr[1][3])};
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const int mi = lane >> 3;
                        const int row = row0 + ((mi & 1) << 3) + (lane & 7);
                        uint32_t w[4];
                        ldmatrix_x4_trans(vb + plane_off<TT, PR, GM>(row, 2 * kk + (mi >> 1)), w[0], w[1], w[2], w[3]);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // granule 2kk + h: words 2h (tokens 0-7), 2h+1 (8-15)
                            uint32_t e0, o0, e1, o1;
                            fp8x4_pairs_to_f16x2<KV>(w[2 * h], e0, o0);
                            fp8x4_pairs_to_f16x2<KV>(w[2 * h + 1], e1, o1);
                            mma_f16_16816(o[4 * kk + 2 * h], pa, e0, e1);
                            mma_f16_16816(o[4 * kk + 2 * h + 1], pa, o0, o1);
                        }
                    }
                }
            }
            if (TMA_KV && partial)
                fence_proxy_async_smem();  // the zeros precede the next TMA into this stage
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&empty_bar[s]));
        }
        if (!ok && lane == 0) {
            record_status(p.status, PKV_ERR_TIMEOUT);
            abort_flag = 1;
        }

        // This CTA's loads are done: the next grid may start its set-up.
        grid_launch_dependents();
        // Merge the compute warps' states (named barrier 1 over the compute threads).
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
        const int r0 = lane >> 2, r1 = r0 + 8;
        if ((lane & 3) == 0) {
            red_m[warp][r0] = m[0];
            red_m[warp][r1] = m[1];
            red_l[warp][r0] = l[0];
            red_l[warp][r1] = l[1];
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");
        if (tid < kDecodeRows) {
            float M = red_m[0][tid];
#pragma unroll
            for (int w = 1; w < NW; ++w)
                M = fmaxf(M, red_m[w][tid]);
            const float ref = M == -INFINITY ? 0.f : M;
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w)
                L += red_l[w][tid] * fast_exp2(red_m[w][tid] - ref);
            row_m[tid] = M;
            // partial states stay unscaled; v_scale goes on the final output
            row_inv_l[tid] = L > 0.f ? (it.partial >= 0 ? 1.f : p.v_scale) / L : 0.f;
            if (tid < it.nheads && !abort_flag) {
                const float lse_v = L > 0.f ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
                const int h = it.head0 + tid;
                if (it.partial >= 0)
                    p.partial_lse[(size_t)it.partial * p.num_qo_heads + h] = lse_v;
                else if (p.lse)
                    p.lse[(size_t)rq.qo_begin * p.num_qo_heads + h] = lse_v;
            }
        }
        // Every stage has been consumed (or the CTA is aborting): the ring holds no
        // copy in flight that is still needed and becomes the combine buffer once
        // all compute warps passed their last tile.
        asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");
        float *sO = reinterpret_cast<float *>(ring_gen);
        {
            const float M0 = row_m[r0], M1 = row_m[r1];
            const float f0 = fast_exp2(m[0] - (M0 == -INFINITY ? 0.f : M0)) * row_inv_l[r0];
            const float f1 = fast_exp2(m[1] - (M1 == -INFINITY ? 0.f : M1)) * row_inv_l[r1];
            if (!KV8) {
                float *w0 = sO + (warp * kDecodeRows + r0) * Tr::kORowFloats + 2 * (lane & 3);
                float *w1 = sO + (warp * kDecodeRows + r1) * Tr::kORowFloats + 2 * (lane & 3);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    *reinterpret_cast<float2 *>(w0 + 8 * i) = make_float2(o[i][0] * f0, o[i][1] * f0);
                    *reinterpret_cast<float2 *>(w1 + 8 * i) = make_float2(o[i][2] * f1, o[i][3] * f1);
                }
            } else {
                // o[2g][e], o[2g+1][e] hold columns 16g + 4c + {0, 2} and {1, 3} (c = lane & 3)
                float *w0 = sO + (warp * kDecodeRows + r0) * Tr::kORowFloats + 4 * (lane & 3);
                float *w1 = sO + (warp * kDecodeRows + r1) * Tr::kORowFloats + 4 * (lane & 3);
#pragma unroll
                for (int g = 0; g < D / 16; ++g) {
                    *reinterpret_cast<float4 *>(w0 + 16 * g) =
                        make_float4(o[2 * g][0] * f0, o[2 * g + 1][0] * f0, o[2 * g][1] * f0, o[2 * g + 1][1] * f0);
                    *reinterpret_cast<float4 *>(w1 + 16 * g) =
                        make_float4(o[2 * g][2] * f1, o[2 * g + 1][2] * f1, o[2 * g][3] * f1, o[2 * g + 1][3] * f1);
                }
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");
        if (!abort_flag) {
            for (int idx = tid; idx < kDecodeRows * (D / 8); idx += NT) {
                const int r = idx / (D / 8);
                const int c = (idx % (D / 8)) * 8;
                if (r >= it.nheads)
                    continue;
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[e] = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float4 *src =
                        reinterpret_cast<const float4 *>(sO + (w * kDecodeRows + r) * Tr::kORowFloats + c);
                    const float4 x = src[0], y = src[1];
                    acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
                    acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
                }
                const int h = it.head0 + r;
                if (it.partial >= 0) {
                    float4 *dst = reinterpret_cast<float4 *>(p.partial_o +
                                                             ((size_t)it.partial * p.num_qo_heads + h) * D + c);
                    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                } else {
                    uint4 v;
                    v.x = pack_bf16(acc[0], acc[1]);
                    v.y = pack_bf16(acc[2], acc[3]);
                    v.z = pack_bf16(acc[4], acc[5]);
                    v.w = pack_bf16(acc[6], acc[7]);
                    *reinterpret_cast<uint4 *>(p.out + ((size_t)rq.qo_begin * p.num_qo_heads + h) * D + c) = v;
                }
            }
        }
        if (it.partial >= 0 && p.merge_counters) {
            // Split-KV: the last CTA of this (request, KV head, head block) group to
            // finish merges the group's partial states through their LSE (the
            // merge_state of the sglang flashinfer_backend.py page, n-way) and re-arms the
            // counter.
            __shared__ int last_flag;
            asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");  // this CTA's partials are written
            if (tid == 0) {
                __threadfence();
                last_flag = atomicAdd(p.merge_counters + it.counter, 1) == it.nsplit - 1;
            }
            asm volatile("bar.sync 1, %0;\n" ::"n"(NT) : "memory");
            if (last_flag) {
                __threadfence();
                constexpr int CPT = D / 8;  // columns per thread: 8 threads per head
                for (int idx = tid; idx < kDecodeRows * 8; idx += NT) {
                const int r = idx >> 3, c0 = (idx & 7) * CPT;
                if (r < it.nheads) {
                    const int h = it.head0 + r;
                    float mx = -INFINITY;
                    for (int k = 0; k < it.nsplit; ++k)
                        mx = fmaxf(mx, __ldcg(p.partial_lse + (size_t)(it.pbase + k) * p.num_qo_heads + h));
                    float acc[CPT];
#pragma unroll
                    for (int e = 0; e < CPT; ++e)
                        acc[e] = 0.f;
                    float sum = 0.f;
                    if (mx != -INFINITY) {
                        for (int k = 0; k < it.nsplit; ++k) {
                            const size_t slot = (size_t)(it.pbase + k) * p.num_qo_heads + h;
                            const float wgt = fast_exp2((__ldcg(p.partial_lse + slot) - mx) * 1.4426950408889634f);
                            const float4 *src = reinterpret_cast<const float4 *>(p.partial_o + slot * D + c0);
#pragma unroll
                            for (int q4 = 0; q4 < CPT / 4; ++q4) {
                                const float4 x = __ldcg(src + q4);
                                acc[4 * q4 + 0] += wgt * x.x;
                                acc[4 * q4 + 1] += wgt * x.y;
                                acc[4 * q4 + 2] += wgt * x.z;
                                acc[4 * q4 + 3] += wgt * x.w;
                            }
                            sum += wgt;
                        }
                    }
                    const float inv = sum > 0.f ? p.v_scale / sum : 0.f;
                    uint16_t *dst = p.out + ((size_t)rq.qo_begin * p.num_qo_heads + h) * D + c0;
#pragma unroll
                    for (int q8 = 0; q8 < CPT / 8; ++q8) {
                        uint4 v;
                        v.x = pack_bf16(acc[8 * q8 + 0] * inv, acc[8 * q8 + 1] * inv);
                        v.y = pack_bf16(acc[8 * q8 + 2] * inv, acc[8 * q8 + 3] * inv);
                        v.z = pack_bf16(acc[8 * q8 + 4] * inv, acc[8 * q8 + 5] * inv);
                        v.w = pack_bf16(acc[8 * q8 + 6] * inv, acc[8 * q8 + 7] * inv);
                        reinterpret_cast<uint4 *>(dst)[q8] = v;
                    }
                    if (p.lse && (idx & 7) == 0)
                        p.lse[(size_t)rq.qo_begin * p.num_qo_heads + h] =
                            sum > 0.f ? mx + __log2f(sum) * 0.6931471805599453f : -INFINITY;
                }
                }
                if (tid == 0)
                    atomicExch(p.merge_counters + it.counter, 0);
            }
        }
    }
}

template <int D, bool TMA_KV, int TT, int KV, int TPW = 16>
cudaError_t launch_decode_dt(const DecodeParams &p, const CUtensorMap &tk, const CUtensorMap &tv, int num_items,
                             cudaStream_t s, bool overlap_prev)
{
    using Tr = DecTraits<D, TT, KV, TPW>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, TMA_KV, TT, KV, TPW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kDynSmem);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    // Programmatic stream serialisation (overlap_prev): this grid's set-up (barriers,
    // work item) may overlap the tail of the previous kernel in the stream; the kernel
    // waits for that kernel's completion before it touches q, the caches or the page
    // table. Not when the previous kernel writes the work list itself.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)num_items);
    cfg.blockDim = dim3(Tr::kThreads);
    cfg.dynamicSmemBytes = Tr::kDynSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap_prev ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_kernel<D, TMA_KV, TT, KV, TPW>, p, tk, tv);
}

}  // namespace dec
}  // namespace pkv
