// Paged prefill / extend kernel on the 5th-generation tensor cores: for head_dim
// 64 and 128 two 128-row query tiles per work item ping-pong over 128-key tiles;
// for head_dim 256 (whose O accumulator takes half of TMEM) one query tile per
// work item runs over 64-key tiles.
//
// Method: plan-clipped KV tiles (the tile-granular KV-start skip of sglang PR
// #31501), the exact per-element mask on boundary tiles, fp32 online softmax with
// lazily rescaled O. Laid out for throughput:
//   * persistent: one CTA per SM walks its own list of work items (balanced by the
//     plan), so TMEM allocation, barrier set-up and the K/V ring are paid once per
//     CTA, the next item's Q and first K/V tiles land while the current item
//     finishes, and an item's epilogue overlaps the next item's first S = Q K^T;
//   * two query tiles Q0, Q1 (256 packed rows) share every K/V tile, halving K/V
//     traffic per flop (head_dim 64 and 128);
//   * P is written back into TMEM over the first half of its own S columns (bf16,
//     two per column) and consumed by tcgen05.mma with the A operand in TMEM, so no
//     shared memory is spent on P;
//   * K and V tiles stream through a ring of 5 (head_dim 128, 256) or 8 (head_dim
//     64) shared-memory slots. Paged bf16 caches use group-major slots (8-key groups
//     of every 64-column chunk): a page of a multiple of 8 keys that divides the
//     KV tile (or is a multiple of it) arrives as ONE 5-D TMA box carrying all its
//     columns, the boxes of a tile spread over three producer warps (one thread
//     issues a TMA box only every 100+ cycles); other page sizes are gathered by
//     cp.async. Q arrives by TMA (4-D map over [token, KV head, group, d]);
//   * one thread issues, per KV tile j: S0(j) = Q0 K_j^T, O1 += P1(j-1) V_{j-1},
//     S1(j) = Q1 K_j^T, O0 += P0(j) V_j, so the tensor core works on one query
//     tile while the softmax warpgroup of the other runs. Tensor-core operations of
//     one thread execute in issue order, which makes S_i(j) complete only after
//     O_i += P_i(j-1) V, the ordering every TMEM reuse below relies on;
//   * one query tile (head_dim 256, bf16 caches): S is double-buffered in TMEM and
//     S(j+1) is issued before O += P(j) V(j), Q is the A operand from TMEM (written
//     by the otherwise idle second warpgroup), and the output of a full item leaves
//     through the Q tile's shared memory as one TMA store per 64-column chunk.
// Warps (384 threads): 0-3 softmax + epilogue of Q0, 4-7 of Q1 (thread = TMEM
// lane = packed row; with one query tile, 4-7 write Q into TMEM), 8 TMEM
// allocation, Q loads and MMA issue (one lane), 9-11 K/V producers (TMA or
// cp.async).
// Every wait is bounded by the plan's wait bound (2 s by default): on expiry
// PKV_ERR_TIMEOUT, abort flag, copies and MMAs drained, TMEM freed.
//
// 8-bit K/V caches (E4M3 / E5M2): warps 9-11 copy the 8-bit rows with cp.async into a
// two-tile staging area and widen them to f16 into the ring; both MMAs run on f16
// operands (every E4M3 / E5M2 value is exact in f16). Each softmax warpgroup writes
// its own Q tile for the next item as f16 with every row scaled by a power of two
// (max |q| * 2^e in [2^13, 2^14)) and scales that row's logits back by 2^-e; P goes to
// the PV MMA as f16.
#pragma once

#include <cfloat>
#include <climits>

#include "pkv_internal.h"
#include "pkv_sm100.cuh"

namespace pkv {
namespace pp {

template <int D, bool KV8 = false>
struct PPTraits {
    static constexpr int kM = 128;            // packed rows per query tile
    static constexpr int kT = D >= 256 ? 64 : 128;  // KV tokens per tile
    static constexpr int kNQ = D >= 256 ? 1 : 2;    // query tiles per CTA (TMEM: S_i, O_i)
    static constexpr int kChunk = 128;        // bytes per swizzled row
    static constexpr int kNCh = D / 64;       // 64-column chunks
    static constexpr int kQTileBytes = kM * D * 2;
    static constexpr int kSlotBytes = kT * D * 2;
    // One query tile over bf16 caches (head_dim 256): Q is the A operand of S = Q K^T
    // from TMEM (128 columns of bf16 pairs), written there from global memory by the
    // second warpgroup, and the Q tile's shared memory stages the bf16 output of the
    // item for one TMA store per 64-column chunk.
    static constexpr bool kQTmem = kNQ == 1 && !KV8;
    // 8-bit caches: fewer f16 slots, and two staging tiles of 8-bit K and V rows.
    static constexpr int kSlots = KV8 ? (D == 64 ? 6 : 3) : (D == 64 ? 8 : 5);
    static constexpr int kStgTileBytes = KV8 ? 2 * kT * D : 0;  // K rows, then V rows
    static constexpr int kOffQ = 0;
    static constexpr int kOffSlots = kNQ * kQTileBytes;
    static constexpr int kOffStg = kOffSlots + kSlots * kSlotBytes;
    static constexpr int kDynSmem = kOffStg + 2 * kStgTileBytes + 1024;
    static constexpr int kThreads = 384;
    static constexpr int kProducers = 96;     // cp.async mode: warps 9-11
    static constexpr int kIdsPerTile = kT;    // page-id ring entries per tile (one per row)
    static constexpr int kTmemCols = 512;
    static constexpr int kTmemO = 256;        // O_i at kTmemO + i * D; S_i at i * kT
    static constexpr int kTmemQ = 2 * kT;     // Q in TMEM (kQTmem): D / 2 columns after the two S buffers
    static_assert(kTmemO + kNQ * D <= kTmemCols && kNQ * kT <= kTmemO, "TMEM budget");
    static_assert(!kQTmem || kTmemQ + D / 2 <= kTmemO, "TMEM budget with Q");
};

// Page-id ring of the cp.async producers, in tiles (ids of kIdRing - 1 tiles in flight).
constexpr int kIdRing = 3;

// K and V of a KV tile complete one barrier, the K slot's: a slot's barrier then
// completes one phase per use of the slot as a K slot. K tiles sit at the even
// ring positions, so with an even slot count every use of an even slot is a K use
// (a phase every NS positions) and with an odd count every other use is (a phase
// every 2 NS positions).
template <int NS>
__host__ __device__ constexpr int full_period() { return NS % 2 == 0 ? NS : 2 * NS; }
constexpr int kRegsLaunch = 168;   // 65536 / 384 rounded down to a multiple of 8
constexpr int kRegsSoftmax = 200;
constexpr int kRegsOther = 96;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= 384 * kRegsLaunch, "register split");

template <int NS>
struct PPBars {
    static constexpr int kQ = 0;
    static constexpr int kFull = 1;              // NS: K and V of a tile landed (on the K slot's barrier)
    static constexpr int kEmpty = kFull + NS;
    static constexpr int kSFull = kEmpty + NS;   // 2: S_i(j) complete in TMEM
    static constexpr int kPFull = kSFull + 2;    // 2: P_i(j) written to TMEM (128 arrivals)
    static constexpr int kOFinal = kPFull + 2;   // 2: O_i of the item complete
    static constexpr int kOEmpty = kOFinal + 2;  // 2: O_i read out by the epilogue (128 arrivals)
    static constexpr int kVLand = kOEmpty + 2;   // producer only: a tail V tile has landed
    static constexpr int kDrain = kVLand + 1;
    static constexpr int kQ1 = kDrain + 1;       // 8-bit caches: Q_1 written (128 arrivals; kQ: Q_0)
    static constexpr int kNever = kQ1 + 1;       // the wait probe's barrier: nothing completes it
    static constexpr int kPVDone = kNever + 1;   // one query tile, S double-buffered: a P V completed
    static constexpr int kQFree = kPVDone + 1;   // Q in TMEM: the item's last S MMA completed
    static constexpr int kOFree = kQFree + 1;    // staged output: the previous item's stores read the tile
    static constexpr int kOStg = kOFree + 1;     // staged output: the item's rows written (128 arrivals)
    static constexpr int kCount = kOStg + 1;
};

template <int D, int MASK, bool TMA_KV, bool RAGGED, int KV = PKV_BF16>
__global__ void __launch_bounds__(384, 1)
    prefill_pp_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o)
{
    constexpr bool KV8 = KV != PKV_BF16;
    static_assert(!KV8 || (!TMA_KV && !RAGGED), "8-bit caches are gathered by the cp.async producers");
    using Tr = PPTraits<D, KV8>;
    constexpr int NS = Tr::kSlots;
    using B = PPBars<NS>;
    constexpr int kFullPeriod = full_period<NS>();
    constexpr int T = Tr::kT;
    constexpr int NCH = Tr::kNCh;
    constexpr int CH = D / 8;
    constexpr bool kCausal = MASK == kMaskCausal || MASK == kMaskCausalWindow;
    constexpr bool kWindow = MASK == kMaskCausalWindow || MASK == kMaskWindow;
    // One query tile per item (head_dim 256, bf16 caches): S is double-buffered in TMEM
    // (S(j+1) is computed while the softmax works on S(j)); the softmax warpgroup is 0.
    constexpr bool kDS = Tr::kNQ == 1 && !KV8;
    // With TMA page boxes, warpgroup 1 writes Q into TMEM (the S MMAs' A operand) and
    // full items' outputs leave through the Q tile's shared memory. With cp.async
    // gathers, warpgroup 1 gathers K/V beside warps 9-11 instead (224 producers: the
    // row gather, not the tensor core, bounds that case), Q stays in shared memory.
    constexpr bool kQTM = kDS && TMA_KV;
    constexpr bool kWideGather = kDS && !TMA_KV;
    constexpr int kGP = kWideGather ? 224 : Tr::kProducers;  // cp.async gather threads
    // Ring slot layout. Paged bf16 caches: group-major, [T/8 key groups][NCH column
    // chunks][8 keys][128 B] (one 1 KB swizzle atom per group and chunk), so that one TMA
    // box of a page carries every column chunk of its rows. Otherwise chunk-major,
    // [NCH][T keys][128 B]. Both are canonical 128-byte-swizzled tcgen05 operand layouts:
    // K is read K-major (8-key groups kGroupStride apart), V MN-major (column chunks
    // kChunkStride apart, 8-key groups kGroupStride apart).
    constexpr bool kGM = !RAGGED && !KV8;
    constexpr uint32_t kChunkStride = kGM ? 1024u : (uint32_t)T * Tr::kChunk;
    constexpr uint32_t kGroupStride = kGM ? (uint32_t)NCH * 1024u : 1024u;
    // byte offset of row t's 128-byte line of column chunk c within a slot (unswizzled)
    auto slot_line = [](int t, int c) -> uint32_t {
        return kGM ? (uint32_t)(t >> 3) * kGroupStride + (uint32_t)c * 1024u + (uint32_t)(t & 7) * 128u
                   : (uint32_t)c * kChunkStride + (uint32_t)t * 128u;
    };

    extern __shared__ uint8_t dsmem_raw[];
    __shared__ __align__(8) uint64_t bars[B::kCount];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    __shared__ int no_abort;
    __shared__ int id_ring[(TMA_KV || KV8) ? 1 : kIdRing * Tr::kIdsPerTile];

    const uint32_t base = (smem_u32(dsmem_raw) + 1023u) & ~1023u;
    const uint32_t sQ = base + Tr::kOffQ;
    const uint32_t sSlots = base + Tr::kOffSlots;
    const uint32_t sStg = base + Tr::kOffStg;  // 8-bit caches only
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    auto slot = [&](int s) { return sSlots + (uint32_t)s * Tr::kSlotBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // After an abort, the TMA producers wait (bounded, ignoring the abort flag) for the
    // K/V tiles whose K went out in the last NS ring positions before n_end, so that no
    // bulk copy lands in shared memory after the CTA has left.
    auto drain_tma_tiles = [&](uint32_t n_end) {
        const uint32_t first = n_end > (uint32_t)NS ? n_end - NS : 0u;
        for (uint32_t nk = first + (first & 1u); nk < n_end; nk += 2)
            mbar_wait(bar(B::kFull + nk % NS), (nk / kFullPeriod) & 1, &no_abort, p.wait_ns);
    };
    // This CTA's work items, in order (the plan balances the lists over the CTAs).
    const int item_lo = p.cta_items[blockIdx.x];
    const int item_hi = p.cta_items[blockIdx.x + 1];
    const int g = p.group;
    const int tq = p.tokens_per_tile;  // query tokens per 128-row tile
    auto q_tiles = [&](const PrefillItem &it) { return (Tr::kNQ > 1 && it.ntok > tq) ? 2 : 1; };
    const volatile int *abort_v = &abort_flag;

    if (threadIdx.x == 0) {
        mbar_init(bar(B::kQ), (KV8 || kQTM) ? 128 : 1);
        mbar_init(bar(B::kQ1), 128);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B::kFull + s), TMA_KV ? 1 : kGP);
            mbar_init(bar(B::kEmpty + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B::kSFull + i), 1);
            mbar_init(bar(B::kPFull + i), 128);
            mbar_init(bar(B::kOFinal + i), 1);
            mbar_init(bar(B::kOEmpty + i), 128);
        }
        mbar_init(bar(B::kVLand), 1);
        mbar_init(bar(B::kDrain), 1);
        mbar_init(bar(B::kNever), 1);
        mbar_init(bar(B::kPVDone), 1);
        mbar_init(bar(B::kQFree), 1);
        mbar_init(bar(B::kOFree), 1);
        mbar_init(bar(B::kOStg), 128);
        abort_flag = 0;
        no_abort = 0;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(&tmem_base_s), Tr::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // Register split: the block is launched with 384 x 168 registers (the build
    // checks that ptxas allocated exactly 168); the softmax warpgroups take 200 and
    // the MMA / producer warpgroup gives back down to 96: 256 x 200 + 128 x 96 =
    // 63488 <= 64512.
    if (warp >= 8)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsOther));
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsSoftmax));

    // cp.async producers of bf16 K/V (page sizes TMA boxes do not suit): thread pt of NP
    // (warps 9-11, and with one query tile warpgroup 1 too).
    auto gather = [&](const int pt) {
            // Work unit = one row and kGU consecutive 16-byte granules of one 64-column
            // chunk's 128-byte line (8, or 4 with 224 producers): one page-table lookup feeds
            // kGU copies (fewer instructions per byte than a granule per lane, which measured
            // slower here although its warp instructions read whole lines). Rows past the
            // cache end are zero-filled. The page id of every row is fetched kIdRing - 1
            // tiles ahead into the shared ring by cp.async (the producers never stall on a
            // page-table read); named barrier 1 orders the ring among the producers.
            constexpr int NP = kGP;
            constexpr int kGU = kWideGather ? 4 : 8;
            constexpr int kUPR = CH / kGU;  // units per row
            constexpr int kUnits = T * kUPR;
            int c_ii = item_lo, c_j = 0, c_at = -1;
            PrefillItem c_it{};
            int c_kv_len = 0, c_page_begin = 0;
            uint32_t n_ids = 0;
            auto fetch_ids = [&]() {
                while (c_ii < item_hi) {
                    if (c_at != c_ii) {
                        c_it = p.items[c_ii];
                        const RequestInfo r = p.reqs[c_it.req];
                        c_kv_len = r.kv_len;
                        c_page_begin = r.kv_page_begin;
                        c_at = c_ii;
                    }
                    if (c_j < c_it.kv_tiles)
                        break;
                    ++c_ii;
                    c_j = 0;
                }
                if (c_ii < item_hi) {
                    const int j0 = prefill_kv_key_at(c_it, c_j, T);
                    for (int t = pt; t < T; t += NP) {
                        int *dst = &id_ring[(n_ids % kIdRing) * Tr::kIdsPerTile + t];
                        const int jj = j0 + t;
                        if (jj < c_kv_len) {
                            const int lp = p.page_shift >= 0 ? (jj >> p.page_shift) : jj / p.page_size;
                            cp_async_4(smem_u32(dst), p.kv_indices + c_page_begin + lp);
                        } else {
                            *dst = -1;
                        }
                    }
                }
                cp_async_commit();
                ++c_j;
                ++n_ids;
            };
            auto sync_producers = [] { asm volatile("bar.sync 1, %0;\n" ::"n"(NP) : "memory"); };
            for (int k = 0; k < kIdRing - 1; ++k)
                fetch_ids();
            uint32_t n = 0;    // K/V ring position
            uint32_t n_t = 0;  // tiles gathered so far
            bool okp = true;
            for (int ii = item_lo; okp && ii < item_hi; ++ii) {
                const PrefillItem it = p.items[ii];
                const int n_tiles = it.kv_tiles;
                if (n_tiles <= 0)
                    continue;
                for (int j = 0; okp && j < n_tiles; ++j, ++n_t) {
                    const int j0 = prefill_kv_key_at(it, j, T);
                    sync_producers();  // every producer is done with the ring entry refilled next
                    fetch_ids();
                    cp_async_wait<kIdRing - 1>();
                    sync_producers();  // this tile's ids are visible to all producers
                    const int *ids = &id_ring[(n_t % kIdRing) * Tr::kIdsPerTile];
                    const uint32_t full = bar(B::kFull + n % NS);  // K and V of the tile complete it
                    for (int isv = 0; isv < 2; ++isv, ++n) {
                        const int s = n % NS;
                        const bool w_ok =
                            n < NS || mbar_wait(bar(B::kEmpty + s), ((n / NS) - 1) & 1, abort_v, p.wait_ns);
                        okp = bar_red_and(1, NP, w_ok);  // every producer takes the same way out
                        if (!okp)
                            break;
                        const uint16_t *src = isv ? p.v_cache : p.k_cache;
                        for (int u = pt; u < kUnits; u += NP) {
                            const int t = u / kUPR, q0 = (u % kUPR) * kGU;  // row, first granule
                            const int jj = j0 + t;
                            const int page = ids[t];
                            size_t off = 0;
                            uint32_t bytes = 0;
                            if (page >= 0) {
                                if ((unsigned)page < (unsigned)p.num_pages) {
                                    const int lp = p.page_shift >= 0 ? (jj >> p.page_shift) : jj / p.page_size;
                                    const int sl = jj - lp * p.page_size;
                                    off = (((size_t)page * p.page_size + sl) * p.num_kv_heads + it.kv_head) * D + q0 * 8;
                                    bytes = 16;
                                } else if (isv == 0) {
                                    record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                                }
                            }
                            const uint32_t line = slot(s) + slot_line(t, q0 >> 3);
    #pragma unroll
                            for (int c = 0; c < kGU; ++c)
                                cp_async_16(line + ((((q0 & 7) + c) ^ (t & 7)) << 4), src + off + c * 8, bytes);
                        }
                        if (isv == 1)
                            cp_async_mbar_arrive(full);
                    }
                }
            }
            if (!okp) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
            }
            asm volatile("cp.async.wait_all;\n" ::: "memory");
    };

    if (warp < 8) {
        if (kWideGather && warp >= 4) {
            gather(96 + (threadIdx.x - 128));
        } else if (kQTM && warp >= 4) {
            // ------------------------------------------------------------ Q into TMEM
            // Warpgroup 1 (idle as a softmax group with one query tile) writes each
            // item's Q tile into TMEM, thread = lane = packed row (token r / g, head
            // r % g): the row's bf16 values as pairs, the A-operand layout of
            // S = Q K^T; rows past the item's tokens are zero. The row travels in two
            // halves of D / 4 words: the next item's first half is loaded from global
            // memory while the current item runs. A tile is stored once the previous
            // item's last S MMA has completed (kQFree); then kQ lets the S MMAs start.
            const int r = threadIdx.x & 127;
            const uint32_t tQ = tmem + ((uint32_t)((warp & 3) * 32) << 16) + Tr::kTmemQ;
            auto next_q_item = [&](int ii) {
                while (ii < item_hi && p.items[ii].kv_tiles <= 0)
                    ++ii;
                return ii;
            };
            auto row_src = [&](int qi) -> const uint4 * {
                const PrefillItem qit = p.items[qi];
                if (r >= qit.ntok * g)
                    return nullptr;
                return reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)(p.reqs[qit.req].qo_begin + qit.tok0 + r / g) * p.num_qo_heads + qit.kv_head * g +
                           r % g) * D);
            };
            bool okq = true;
            uint32_t n_st = 0;  // Q tiles stored: the phase of kQFree
            int qi = next_q_item(item_lo);
            const uint4 *src = qi < item_hi ? row_src(qi) : nullptr;
            uint4 hv[D / 16];
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                hv[k] = src ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
            while (qi < item_hi) {
                if (n_st > 0) {
                    okq = __all_sync(0xffffffffu, mbar_wait(bar(B::kQFree), (n_st - 1) & 1, abort_v, p.wait_ns));
                    if (!okq)
                        break;
                    tc_fence_after();
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
                    for (int c = 0; c < D / 128; ++c) {
                        uint32_t w[32];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const uint4 v = hv[8 * c + e];
                            w[4 * e + 0] = v.x;
                            w[4 * e + 1] = v.y;
                            w[4 * e + 2] = v.z;
                            w[4 * e + 3] = v.w;
                        }
                        tmem_st32u(tQ + hf * (D / 4) + 32 * c, w);
                    }
                    if (hf == 0) {
#pragma unroll
                        for (int k = 0; k < D / 16; ++k)
                            hv[k] = src ? __ldg(src + D / 16 + k) : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(B::kQ));
                ++n_st;
                qi = next_q_item(qi + 1);
                src = qi < item_hi ? row_src(qi) : nullptr;
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    hv[k] = src ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (!okq) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
            }
        } else {
            // ------------------------------------------------------------ softmax
            const int wg = warp >> 2;
            const int r = threadIdx.x & 127;
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + lane_off + wg * T;
            const uint32_t tO = tmem + lane_off + Tr::kTmemO + wg * D;
            float scale = p.sm_scale_log2;  // raw dot (or capped logit) -> log2-domain logit
            float cap_in = p.cap_in;         // raw dot -> tanh argument
            uint32_t n_s = 0;  // S_wg tiles consumed so far: the phase of SFull / PFull
            uint32_t n_o = 0;  // items accumulated into O_wg so far: the phase of OFinal / OEmpty
            uint32_t n_stg = 0;  // items whose output went through shared memory: the phase of kOFree / kOStg
            bool ok = true;
            // 8-bit caches: the next item whose Q_wg this warpgroup writes (an item with
            // KV tiles that uses query tile wg), and the scale-back of this thread's row.
            auto next_q_item = [&](int ii) {
                while (ii < item_hi && (p.items[ii].kv_tiles <= 0 || wg >= q_tiles(p.items[ii])))
                    ++ii;
                return ii;
            };
            // Row r of Q_wg for item qi: q scaled by 2^e (e from the row's max |q|), as f16,
            // in the 128-byte-swizzled K-major layout of the S MMA's A operand; rows past
            // the item's tokens are zero. Q_wg is free: the S_wg MMAs of the previous item,
            // its only readers, completed before their last S was consumed.
            auto write_q = [&](int qi) -> float {
                const PrefillItem qit = p.items[qi];
                const int nt = min(tq, qit.ntok - wg * tq);
                const bool valid = r < nt * g;
                const int tok = qit.tok0 + wg * tq + r / g;
                const int h = qit.kv_head * g + r % g;
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)(p.reqs[qit.req].qo_begin + (valid ? tok : 0)) * p.num_qo_heads + h) * D);
                float amax = 0.f;
                if (valid) {
    #pragma unroll 4
                    for (int k = 0; k < D / 8; ++k) {
                        const uint4 v = __ldg(src + k);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
                        for (int e = 0; e < 4; ++e)
                            amax = max3f(amax, fabsf(__uint_as_float(w4[e] << 16)),
                                         fabsf(__uint_as_float(w4[e] & 0xffff0000u)));
                    }
                }
                int qe = 13 - ((int)((__float_as_uint(amax) >> 23) & 0xff) - 127);
                qe = qe < -100 ? -100 : (qe > 100 ? 100 : qe);
                const float up = __uint_as_float((uint32_t)(127 + qe) << 23);
                const uint32_t qtile = sQ + wg * Tr::kQTileBytes;
    #pragma unroll 4
                for (int k = 0; k < D / 8; ++k) {
                    const uint4 v = valid ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    uint32_t f[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e)
                        f[e] = pack_f16(__uint_as_float(w4[e] << 16) * up, __uint_as_float(w4[e] & 0xffff0000u) * up);
                    const uint32_t a = qtile + (k >> 3) * (128 * Tr::kChunk) + r * Tr::kChunk + (((k & 7) ^ (r & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(f[0]), "r"(f[1]), "r"(f[2]),
                                 "r"(f[3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(wg == 0 ? B::kQ : B::kQ1));
                return __uint_as_float((uint32_t)(127 - qe) << 23);
            };
            int q_item = item_hi;
            float q_unscale = 1.f;
            if (KV8) {
                q_item = next_q_item(item_lo);
                if (q_item < item_hi)
                    q_unscale = write_q(q_item);
            }
            for (int ii = item_lo; ok && ii < item_hi; ++ii) {
                const PrefillItem it = p.items[ii];
                if (wg >= q_tiles(it))
                    continue;
                if (KV8 && it.kv_tiles > 0) {
                    // this item is q_item: its logits carry the row's 2^e
                    scale = p.cap_in > 0.f ? p.sm_scale_log2 : p.sm_scale_log2 * q_unscale;
                    cap_in = p.cap_in * q_unscale;
                }
                const RequestInfo rq = p.reqs[it.req];
                const int n_tiles = it.kv_tiles;
                const int ntok_wg = min(tq, it.ntok - wg * tq);
                const int tok = it.tok0 + wg * tq + r / g;
                const int pos = rq.q_start + tok;
                const int p_min = rq.q_start + it.tok0 + wg * tq;
                const int p_max = p_min + ntok_wg - 1;
                float m_used = -INFINITY;
                float l = 0.f;
                for (int j = 0; j < n_tiles; ++j, ++n_s) {
                    // double-buffered S: tile n_s sits in buffer n_s & 1 (barriers SFull / PFull + buffer)
                    const int sb = kDS ? (int)(n_s & 1) : wg;
                    const uint32_t sphase = kDS ? (n_s >> 1) & 1 : n_s & 1;
                    const uint32_t tSb = kDS ? tmem + lane_off + sb * T : tS;
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull + sb), sphase, abort_v, p.wait_ns));
                    if (!ok)
                        break;
                    tc_fence_after();
                    float s[T];
    #pragma unroll
                    for (int c = 0; c < T / 32; ++c)
                        tmem_ld32(tSb + 32 * c, *reinterpret_cast<float(*)[32]>(&s[32 * c]));
                    tmem_wait_ld();
                    if (p.cap_in > 0.f) {
                        // soft cap on the raw dot products, before the mask
    #pragma unroll
                        for (int c = 0; c < T; ++c)
                            s[c] = p.cap_out * soft_cap_tanh(s[c] * cap_in);
                    }

                    const int j0 = prefill_kv_key_at(it, j, T);
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
                            s[c] = (c >= lo_c && c <= hi_c) ? s[c] : -INFINITY;
                    }
                    // 8 independent chains of three-input maxima, then a tree: the row
                    // max costs T/2 instructions and stays off a long dependency chain.
                    float mx8[8];
    #pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mx8[k] = max3f(s[k], s[k + 8], s[k + 16]);
    #pragma unroll
                    for (int c = 24; c + 16 <= T; c += 16)
    #pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mx8[k] = max3f(mx8[k], s[c + k], s[c + 8 + k]);
    #pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mx8[k] = fmaxf(mx8[k], s[T - 8 + k]);
                    const float m_raw = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                                              fmaxf(mx8[6], mx8[7]));
                    const float m_tile = m_raw == -INFINITY ? -INFINITY : m_raw * scale;
                    const float m_cand = fmaxf(m_used, m_tile);
                    const bool need = m_cand != -INFINITY && (m_used == -INFINITY || m_cand > m_used + 8.f);
                    const float alpha = need ? fast_exp2(m_used - m_cand) : 1.f;
                    if (j > 0 && __any_sync(0xffffffffu, need)) {
                        // O_i is stable: S_i(j) completed after O_i += P_i(j-1) V. With S
                        // double-buffered, S(j) was issued before P(j-1) V: wait for it.
                        if (kDS) {
                            ok = __all_sync(0xffffffffu,
                                            mbar_wait(bar(B::kPVDone), (n_s - 1) & 1, abort_v, p.wait_ns));
                            if (!ok)
                                break;
                            tc_fence_after();
                        }
    #pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            tmem_ld32(tO + 32 * c, o);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] *= alpha;
                            tmem_st32(tO + 32 * c, o);
                        }
                    }
                    if (need) {
                        l *= alpha;
                        m_used = m_cand;
                    }
                    const float nref = -(m_used == -INFINITY ? 0.f : m_used);
                    // Packed f32x2 arithmetic: one FMA and one add per two scores.
                    float rs[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    #pragma unroll
                    for (int h = 0; h < T / 64; ++h) {
                        uint32_t pw[32];
    #pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            float x0, x1;
                            fma2(x0, x1, s[64 * h + 2 * k], s[64 * h + 2 * k + 1], scale, scale, nref, nref);
                            const float e0 = fast_exp2(x0);
                            const float e1 = fast_exp2(x1);
                            add2(rs[k & 3][0], rs[k & 3][1], e0, e1);
                            pw[k] = KV8 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
                        }
                        tmem_st32u(tSb + 32 * h, pw);
                    }
                    tmem_wait_st();
                    l += ((rs[0][0] + rs[0][1]) + (rs[1][0] + rs[1][1])) + ((rs[2][0] + rs[2][1]) + (rs[3][0] + rs[3][1]));
                    tc_fence_before();
                    mbar_arrive(bar(B::kPFull + sb));
                }
                if (KV8 && ok && n_tiles > 0) {
                    // Every S_wg of this item has been consumed: Q_wg of the next item may be
                    // written now, so that its first S MMA overlaps this item's epilogue.
                    q_item = next_q_item(ii + 1);
                    if (q_item < item_hi)
                        q_unscale = write_q(q_item);
                }
                if (ok && n_tiles > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kOFinal + wg), n_o & 1, abort_v, p.wait_ns));
                    tc_fence_after();
                }
                if (!ok)
                    break;
                const bool row_ok = r < ntok_wg * g;
                const int h = it.kv_head * g + r % g;
                const size_t orow = (size_t)(rq.qo_begin + tok) * p.num_qo_heads + h;
                uint16_t *dst = p.out + orow * D;
                const float inv = l > 0.f ? p.v_scale / l : 0.f;
                // One query tile of full items: the bf16 rows go through the Q tile's
                // shared memory, in the layout of the output tensor map's boxes, and
                // leave as one TMA store per 64-column chunk (whole lines, where a
                // thread-per-row store would touch 32 lines per instruction).
                const bool staged = kQTM && n_tiles > 0 && ntok_wg == tq;
                if (staged) {
                    if (r == 0) {
                        bulk_wait_read0();  // the previous item's stores have read the tile
                        mbar_arrive(bar(B::kOFree));
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kOFree), n_stg & 1, abort_v, p.wait_ns));
                    if (!ok)
                        break;
                }
    #pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    if (n_tiles > 0) {
                        tmem_ld32(tO + 32 * c, o);
                        tmem_wait_ld();
                    } else {
    #pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = 0.f;
                    }
                    if (staged) {
    #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const uint32_t a = sQ + (c >> 1) * (128 * Tr::kChunk) + r * Tr::kChunk +
                                               ((((c & 1) * 4 + q4) ^ (r & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a),
                                         "r"(pack_bf16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv)),
                                         "r"(pack_bf16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv)),
                                         "r"(pack_bf16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv)),
                                         "r"(pack_bf16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv))
                                         : "memory");
                        }
                    } else if (row_ok) {
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
                if (staged) {
                    fence_proxy_async_smem();  // the rows are read by the TMA stores
                    mbar_arrive(bar(B::kOStg));
                    if (r == 0) {
                        ok = mbar_wait(bar(B::kOStg), n_stg & 1, abort_v, p.wait_ns);
                        if (ok) {
                            for (int cc = 0; cc < NCH; ++cc)
                                tma_store_4d(&tm_o, sQ + cc * (128 * Tr::kChunk), cc * 64, 0, it.kv_head,
                                             rq.qo_begin + it.tok0);
                            bulk_commit();
                        }
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    ++n_stg;
                }
                if (n_tiles > 0) {
                    // O_wg has been read: the next item's first P V may overwrite it.
                    tc_fence_before();
                    mbar_arrive(bar(B::kOEmpty + wg));
                    ++n_o;
                }
                if (row_ok && p.lse)
                    p.lse[orow] = l > 0.f ? (m_used + __log2f(l)) * 0.6931471805599453f : -INFINITY;
            }
            if (!ok) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
            }
            if (kQTM && threadIdx.x == 0)
                bulk_wait0();  // the output stores are done before the CTA leaves
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issue
        // One lane drives everything: Q loads, waits, MMA issue and commits.
        if (lane == 0) {
            const uint32_t idesc_s = KV8 ? idesc_f16_f32(128, T, false) : idesc_bf16_f32(128, T, false);
            const uint32_t idesc_o = KV8 ? idesc_f16_f32(128, D, true) : idesc_bf16_f32(128, D, true);
            auto issue_s = [&](int i, uint32_t kslot) {
                const uint32_t qb = sQ + i * Tr::kQTileBytes;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t a = sdesc_sw128(qb + (k >> 2) * (128 * Tr::kChunk) + (k & 3) * 32, 16, 1024);
                    const uint64_t b = sdesc_sw128(kslot + (k >> 2) * kChunkStride + (k & 3) * 32, 16, kGroupStride);
                    umma_f16(tmem + i * T, a, b, idesc_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(B::kSFull + i));
            };
            auto issue_pv = [&](int i, uint32_t vslot, bool first) {
#pragma unroll
                for (int k = 0; k < T / 16; ++k) {
                    const uint64_t b = sdesc_sw128(vslot + k * 2 * kGroupStride, kChunkStride, kGroupStride);
                    umma_f16_ts(tmem + Tr::kTmemO + i * D, tmem + i * T + k * 8, b, idesc_o,
                                (!first || k > 0) ? 1u : 0u);
                }
            };
            auto wait = [&](int b_idx, uint32_t parity) {
                return mbar_wait(bar(b_idx), parity, abort_v, p.wait_ns);
            };
            // Q of an item: its tiles by TMA (4-D map over [token, KV head, group, d]).
            auto load_q = [&](int ii) {
                const PrefillItem it = p.items[ii];
                const int nq = q_tiles(it);
                const int qo_begin = p.reqs[it.req].qo_begin;
                const uint32_t rows = (uint32_t)(g * tq);
                const uint32_t qbar = bar(B::kQ);
                mbar_arrive_expect_tx(qbar, (uint32_t)nq * NCH * rows * Tr::kChunk);
                for (int i = 0; i < nq; ++i)
                    for (int c = 0; c < NCH; ++c)
                        tma_load_4d(sQ + i * Tr::kQTileBytes + c * (128 * Tr::kChunk), &tm_q, c * 64, 0, it.kv_head,
                                    qo_begin + it.tok0 + i * tq, qbar);
            };
            // The next item at or after ii that has KV tiles (items without any
            // only write zeros and take no part in the pipeline).
            auto next_busy = [&](int ii) {
                while (ii < item_hi && p.items[ii].kv_tiles <= 0)
                    ++ii;
                return ii;
            };
            if (!KV8)
                tma_prefetch_desc(&tm_q);
            uint32_t n_kv = 0;         // K/V ring position
            uint32_t n_p[2] = {0, 0};  // P_i tiles consumed: the phase of PFull_i
            uint32_t n_o[2] = {0, 0};  // items accumulated into O_i: the phase of OEmpty_i
            uint32_t n_q = 0;          // Q loads: the phase of kQ
            uint32_t n_q1 = 0;         // 8-bit caches: Q_1 writes, the phase of kQ1
            bool probe = p.wait_probe != 0;  // the first K/V wait is on a barrier nothing completes
            bool ok = true;
            int ii = next_busy(item_lo);
            if (!KV8 && !kQTM && ii < item_hi)
                load_q(ii);
            // One query tile, S double-buffered: per item, S(0), then for each KV tile j
            // S(j+1) (into the other buffer) before O += P(j) V(j), so that the tensor
            // core computes S(j+1) while the softmax turns S(j) into P(j). In issue
            // order S(j+1) precedes P(j) V: a buffer is rewritten (S(j+2)) only after
            // the P V that read it was issued, and the softmax waits for kPVDone before
            // it rescales O. The next item's Q lands once the item's last S completed.
            uint32_t n_sq = 0;  // S tiles issued: buffer n_sq & 1, its phase (n_sq >> 1) & 1
            uint32_t n_pv = 0;  // P V issued: P in buffer n_pv & 1
            while (kDS && ok && ii < item_hi) {
                const PrefillItem it = p.items[ii];
                const int n_tiles = it.kv_tiles;
                const int ii_next = next_busy(ii + 1);
                if (!(ok = wait(B::kQ, n_q & 1)))
                    break;
                ++n_q;
                // S of the item's tile jj: wait for its K (and V) and issue it
                auto next_s = [&](uint32_t &sv) -> bool {
                    const uint32_t nK = n_kv;
                    n_kv += 2;
                    const int sK = nK % NS;
                    sv = (nK + 1) % NS;
                    if (!wait(probe ? B::kNever : B::kFull + sK, (nK / kFullPeriod) & 1))
                        return false;
                    probe = false;
                    if (!TMA_KV)
                        fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t kslot = slot(sK);
                    const uint32_t dst = tmem + (n_sq & 1) * T;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint64_t b = sdesc_sw128(kslot + (k >> 2) * kChunkStride + (k & 3) * 32, 16, kGroupStride);
                        if (kQTM) {
                            umma_f16_ts(dst, tmem + Tr::kTmemQ + k * 8, b, idesc_s, k > 0 ? 1u : 0u);
                        } else {
                            const uint64_t a = sdesc_sw128(sQ + (k >> 2) * (128 * Tr::kChunk) + (k & 3) * 32, 16, 1024);
                            umma_f16(dst, a, b, idesc_s, k > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(bar(B::kSFull + (n_sq & 1)));
                    umma_commit(bar(B::kEmpty + sK));
                    ++n_sq;
                    return true;
                };
                // the item's last S has completed: Q (in TMEM, or its shared tile) is free
                // for the next item
                auto next_q = [&]() -> bool {
                    const uint32_t m = n_sq - 1;
                    if (!wait(B::kSFull + (m & 1), (m >> 1) & 1))
                        return false;
                    if (kQTM)
                        mbar_arrive(bar(B::kQFree));
                    else
                        load_q(ii_next);
                    return true;
                };
                uint32_t sv_cur = 0, sv_next = 0;
                if (!(ok = next_s(sv_cur)))
                    break;
                if (n_tiles == 1 && ii_next < item_hi && !(ok = next_q()))
                    break;
                for (int j = 0; j < n_tiles; ++j) {
                    if (j + 1 < n_tiles && !(ok = next_s(sv_next)))
                        break;
                    if (!(ok = wait(B::kPFull + (n_pv & 1), (n_pv >> 1) & 1)))
                        break;
                    if (j == 0 && n_o[0] > 0 && !(ok = wait(B::kOEmpty + 0, (n_o[0] - 1) & 1)))
                        break;
                    tc_fence_after();
                    const uint32_t vslot = slot(sv_cur);
#pragma unroll
                    for (int k = 0; k < T / 16; ++k) {
                        const uint64_t b = sdesc_sw128(vslot + k * 2 * kGroupStride, kChunkStride, kGroupStride);
                        umma_f16_ts(tmem + Tr::kTmemO, tmem + (n_pv & 1) * T + k * 8, b, idesc_o,
                                    (j > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(bar(B::kEmpty + sv_cur));
                    umma_commit(bar(B::kPVDone));
                    ++n_pv;
                    if (j == n_tiles - 1)
                        umma_commit(bar(B::kOFinal + 0));
                    if (j + 2 == n_tiles && ii_next < item_hi && !(ok = next_q()))
                        break;
                    sv_cur = sv_next;
                }
                ++n_o[0];
                ii = ii_next;
            }
            while (!kDS && ok && ii < item_hi) {
                const PrefillItem it = p.items[ii];
                const int nq = q_tiles(it);
                const int n_tiles = it.kv_tiles;
                const int ii_next = next_busy(ii + 1);
                if (!(ok = wait(B::kQ, n_q & 1)))
                    break;
                ++n_q;
                if (KV8 && nq == 2) {  // Q_1 is written by its own warpgroup
                    if (!(ok = wait(B::kQ1, n_q1 & 1)))
                        break;
                    ++n_q1;
                }
                uint32_t sv_prev = 0;
                for (int j = 0; j < n_tiles; ++j) {
                    const uint32_t nK = n_kv, nV = n_kv + 1;
                    n_kv += 2;
                    const int sK = nK % NS, sV = nV % NS;
                    // 8-bit caches: K and V complete their own slots' barriers (one phase
                    // per use), so S_0 starts as soon as K is widened, V is waited for
                    // before its first P V.
                    if (!(ok = wait(probe ? B::kNever : B::kFull + sK, (nK / (KV8 ? NS : kFullPeriod)) & 1)))
                        break;
                    probe = false;
                    if (!TMA_KV)
                        fence_proxy_async_smem();
                    tc_fence_after();
                    issue_s(0, slot(sK));
                    if (j > 0 && nq == 2) {
                        if (!(ok = wait(B::kPFull + 1, n_p[1]++ & 1)))
                            break;
                        if (j == 1 && n_o[1] > 0 && !(ok = wait(B::kOEmpty + 1, (n_o[1] - 1) & 1)))
                            break;
                        tc_fence_after();
                        issue_pv(1, slot(sv_prev), j == 1);
                        umma_commit(bar(B::kEmpty + sv_prev));
                    }
                    if (nq == 2)
                        issue_s(1, slot(sK));
                    umma_commit(bar(B::kEmpty + sK));
                    if (!(ok = wait(B::kPFull + 0, n_p[0]++ & 1)))
                        break;
                    if (j == 0 && n_o[0] > 0 && !(ok = wait(B::kOEmpty + 0, (n_o[0] - 1) & 1)))
                        break;
                    tc_fence_after();
                    // Single query tile: S_0 of the last KV tile has been consumed, so
                    // every read of Q is done and the next item's Q may land.
                    if (!KV8 && nq == 1 && j == n_tiles - 1 && ii_next < item_hi)
                        load_q(ii_next);
                    if (KV8) {
                        if (!(ok = wait(B::kFull + sV, (nV / NS) & 1)))
                            break;
                        fence_proxy_async_smem();
                        tc_fence_after();
                    }
                    issue_pv(0, slot(sV), j == 0);
                    if (nq == 1)
                        umma_commit(bar(B::kEmpty + sV));
                    if (j == n_tiles - 1)
                        umma_commit(bar(B::kOFinal + 0));
                    sv_prev = sV;
                }
                if (ok && nq == 2) {
                    ok = wait(B::kPFull + 1, n_p[1]++ & 1);
                    if (ok && n_tiles == 1 && n_o[1] > 0)
                        ok = wait(B::kOEmpty + 1, (n_o[1] - 1) & 1);
                    if (ok) {
                        tc_fence_after();
                        // S_1 of the last KV tile (issued after S_0) has been consumed.
                        if (!KV8 && ii_next < item_hi)
                            load_q(ii_next);
                        issue_pv(1, slot(sv_prev), n_tiles == 1);
                        umma_commit(bar(B::kEmpty + sv_prev));
                        umma_commit(bar(B::kOFinal + 1));
                    }
                }
                ++n_o[0];
                if (nq == 2)
                    ++n_o[1];
                ii = ii_next;
            }
            if (!ok) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
            }
            umma_commit(bar(B::kDrain));
            mbar_wait(bar(B::kDrain), 0, &no_abort, p.wait_ns);
        }
        __syncwarp();
    } else if (RAGGED) {
        // ------------------------------------------------------------ TMA producer, ragged K/V
        // K/V rows of request b are rows kv_page_begin + j of a [total_kv, H_kv, d]
        // tensor: one box per 64-column chunk of a tile, at any row. Rows past the
        // request's keys are the next request's (finite, masked in S, so P = 0) or
        // past the tensor's end (filled with zeros by the copy).
        static_assert(!RAGGED || TMA_KV, "ragged K/V are loaded by TMA");
        if (warp == 9 && lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t n = 0;  // K/V ring position
            bool okp = true;
            for (int ii = item_lo; okp && ii < item_hi; ++ii) {
                const PrefillItem it = p.items[ii];
                const int n_tiles = it.kv_tiles;
                if (n_tiles <= 0)
                    continue;
                const int row_base = p.reqs[it.req].kv_page_begin;
                for (int j = 0; okp && j < n_tiles; ++j) {
                    const int row0 = row_base + prefill_kv_key_at(it, j, T);
                    const uint32_t full = bar(B::kFull + n % NS);  // K and V of the tile complete it
                    for (int isv = 0; isv < 2; ++isv, ++n) {
                        const int s = n % NS;
                        if (n >= NS && !mbar_wait(bar(B::kEmpty + s), ((n / NS) - 1) & 1, abort_v, p.wait_ns)) {
                            okp = false;
                            break;
                        }
                        if (isv == 0)
                            mbar_arrive_expect_tx(full, 2u * T * Tr::kChunk * NCH);
                        const void *tm = isv ? (const void *)&tm_v : (const void *)&tm_k;
                        for (int c = 0; c < NCH; ++c)
                            tma_load_4d(slot(s) + c * (T * Tr::kChunk), tm, c * 64, it.kv_head, row0, 0, full);
                    }
                }
            }
            if (!okp) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
                drain_tma_tiles(n);
            }
        }
    } else if (TMA_KV) {
        // ------------------------------------------------------------ TMA producers
        // Warps 9-11. One 5-D box per page and tile carries every column chunk of the
        // page's rows (rows_box keys = rows_box / 8 key groups of the group-major slot).
        // A tile's 2 npg boxes (K, then V) are spread over the three warps, whose TMA
        // issue runs in parallel (one thread issues a box about every 100+ cycles).
        // The three warps take every ring position in lockstep: each waits for the slot,
        // then a named barrier among them (which also carries an expired wait, or warp
        // 9's failed tail landing, to all three), then warp 9 sets the expected bytes
        // and the boxes go out. A tile's barrier thus completes only after every warp
        // has seen both of its slots free, so no warp can fall a whole phase behind
        // the consumer (a parity wait needs that), whether or not it has a box in the
        // tile (with one box per tile, warp 11 has none). Warp 9 also handles the tail
        // tiles' V rows.
        static_assert(!TMA_KV || RAGGED || kGM, "paged TMA boxes fill the group-major layout");
        const int pw = warp - 9;  // 0, 1, 2
        {
            const int P = p.page_size;
            const int rows_box = P < T ? P : T;
            const int npg = T / rows_box;
            if (lane == 0) {
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
            }
            uint32_t n = 0;       // K/V ring position
            uint32_t n_land = 0;  // tail V tiles so far: the phase of kVLand (warp 9)
            bool okp = true;
            bool land_ok = true;  // warp 9: the last tail V tile landed
            for (int ii = item_lo; okp && ii < item_hi; ++ii) {
                const PrefillItem it = p.items[ii];
                const int n_tiles = it.kv_tiles;
                if (n_tiles <= 0)
                    continue;
                const RequestInfo rq = p.reqs[it.req];
                const int n_pages_req = (rq.kv_len + P - 1) / P;
                // Lane i: the physical page of the tile's i-th box, or -1.
                auto load_id = [&](int j) -> int {
                    if (lane >= npg)
                        return -1;
                    const int j0 = prefill_kv_key_at(it, j, T);
                    const int lp = P <= T ? j0 / P + lane : j0 / P;
                    if (lp >= n_pages_req)
                        return -1;
                    const int pg = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                    if ((unsigned)pg >= (unsigned)p.num_pages) {
                        if (pw == 0)
                            record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                        return -1;
                    }
                    return pg;
                };
                int pg = load_id(0);
                for (int j = 0; okp && j < n_tiles; ++j) {
                    const int j0 = prefill_kv_key_at(it, j, T);
                    const int slot0 = P > T ? j0 % P : 0;
                    int pg_next = -1;
                    // K, then V. Both complete the K slot's barrier; a V tile reaching
                    // past the cache end lands on warp 9's own barrier instead: its rows
                    // past the end hold stale or foreign data and are zeroed (so that
                    // P = 0 never meets a non-finite value) before warp 9's arrival
                    // completes the K slot's barrier.
                    const bool tail = j0 + T > rq.kv_len;
                    const unsigned valid = __ballot_sync(0xffffffffu, pg >= 0);
                    const uint32_t bytes = (uint32_t)__popc(valid) * rows_box * Tr::kChunk * NCH;
                    const uint32_t full = bar(B::kFull + n % NS);
                    for (int isv = 0; isv < 2; ++isv, ++n) {
                        const int s = n % NS;
                        const bool w_ok =
                            n < NS || mbar_wait(bar(B::kEmpty + s), ((n / NS) - 1) & 1, abort_v, p.wait_ns);
                        okp = bar_red_and(1, 96, w_ok && land_ok);
                        if (!okp)
                            break;
                        const bool vtail = isv == 1 && tail;
                        const uint32_t land = vtail ? bar(B::kVLand) : full;
                        if (pw == 0 && lane == 0) {
                            if (isv == 0 && tail)
                                mbar_expect_tx(full, bytes);  // the arrival comes after the zeroing
                            else if (isv == 0)
                                mbar_arrive_expect_tx(full, 2 * bytes);
                            else if (vtail)
                                mbar_arrive_expect_tx(land, bytes);
                        }
                        __syncwarp();
                        // box `lane` of K (isv 0) or V (isv 1), issued by warp (isv npg + lane) % 3;
                        // a tail tile's V boxes all by warp 9 (the others may already be at a
                        // later tile, and kVLand must see one tail tile's bytes at a time)
                        if (pg >= 0 && (vtail ? pw == 0 : (isv * npg + lane) % 3 == pw)) {
                            const void *tm = isv ? (const void *)&tm_v : (const void *)&tm_k;
                            tma_load_5d(slot(s) + (uint32_t)(lane * rows_box / 8) * kGroupStride, tm, 0, 0, 0,
                                        it.kv_head, (pg * P + slot0) >> 3, land);
                        }
                        if (isv == 0 && j + 1 < n_tiles)
                            pg_next = load_id(j + 1);
                        if (vtail && pw == 0) {
                            // (a failed landing reaches the other warps at the next barrier)
                            land_ok = __all_sync(0xffffffffu,
                                                 mbar_wait(bar(B::kVLand), n_land & 1, abort_v, p.wait_ns));
                            ++n_land;
                            if (!land_ok)
                                continue;
                            const int vr = max(0, rq.kv_len - j0);
                            const int n16 = (T - vr) * 8;  // 16-byte granules per chunk
                            for (int idx = lane; idx < n16 * NCH; idx += 32) {
                                const int c = idx / n16, e = idx % n16;
                                const uint32_t a = slot(s) + slot_line(vr + e / 8, c) + (e % 8) * 16;
                                asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};\n" ::"r"(a), "r"(0) : "memory");
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(full);
                        }
                    }
                    pg = pg_next;
                }
            }
            okp = okp && land_ok;
            if (!okp && lane == 0) {
                record_status(p.status, PKV_ERR_TIMEOUT);
                abort_flag = 1;
                if (pw == 0)
                    drain_tma_tiles(n);
            }
        }
    } else if (!KV8) {
        // ------------------------------------------------------------ cp.async producers
        gather(threadIdx.x - 9 * 32);
    } else {
        // ------------------------------------------------------------ 8-bit K/V producers
        // Step n: the 8-bit K and V rows of this CTA's n-th KV tile are copied by
        // cp.async into staging buffer n % 2 (rows past the cache end or behind a bad
        // page id are zero-filled), while the tile staged in step n - 1 is widened to
        // f16 into its ring slots, in the layout the TMA path produces. Each thread's
        // page ids for the next tile are loaded one step ahead.
        constexpr int NP = Tr::kProducers;
        constexpr bool E5 = KV == PKV_FP8_E5M2;
        constexpr int CPR = D / 16;                   // 16-byte chunks per 8-bit row
        constexpr int SWZ = (CPR < 8 ? CPR : 8) - 1;  // chunk swizzle of the staging rows
        constexpr int kUPT = (2 * T + NP - 1) / NP;   // copy units (row, K or V) per thread
        const int pt = threadIdx.x - 9 * 32;
        const uint8_t *kc = reinterpret_cast<const uint8_t *>(p.k_cache);
        const uint8_t *vc = reinterpret_cast<const uint8_t *>(p.v_cache);
        auto sync_producers = [] { asm volatile("bar.sync 1, %0;\n" ::"n"(NP) : "memory"); };
        auto first_from = [&](int ii) {
            while (ii < item_hi && p.items[ii].kv_tiles <= 0)
                ++ii;
            return ii;
        };
        // Page id (-1: no key) and slot of each of this thread's copy units of tile (ii, j).
        auto load_ids = [&](int ii, int j, int (&pg)[kUPT], int (&sl)[kUPT]) {
            const PrefillItem it = p.items[ii];
            const RequestInfo rq = p.reqs[it.req];
            const int j0 = prefill_kv_key_at(it, j, T);
#pragma unroll
            for (int k = 0; k < kUPT; ++k) {
                const int u = pt + k * NP;
                const int jj = j0 + u % T;
                pg[k] = -1;
                sl[k] = 0;
                if (u < 2 * T && jj < rq.kv_len) {
                    const int lp = p.page_shift >= 0 ? (jj >> p.page_shift) : jj / p.page_size;
                    pg[k] = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                    sl[k] = jj - lp * p.page_size;
                }
            }
        };
        int cur_ii = first_from(item_lo), cur_j = 0;
        int pg[kUPT], sl[kUPT];
        if (cur_ii < item_hi)
            load_ids(cur_ii, cur_j, pg, sl);
        uint32_t n = 0;  // ring position of the next tile to widen (K at n, V at n + 1)
        int staged = 0;  // tiles copied so far
        bool okp = true;
        while (true) {
            const bool have = cur_ii < item_hi;
            sync_producers();  // buffer staged % 2 was widened in the previous step by every producer
            if (have) {
                const uint32_t stg = sStg + (uint32_t)(staged & 1) * Tr::kStgTileBytes;
                const int kvh = p.items[cur_ii].kv_head;
#pragma unroll
                for (int k = 0; k < kUPT; ++k) {
                    const int u = pt + k * NP;
                    if (u >= 2 * T)
                        continue;
                    const int t = u % T, isv = u / T;
                    int64_t off = -1;
                    if (pg[k] >= 0) {
                        if ((unsigned)pg[k] < (unsigned)p.num_pages)
                            off = (((int64_t)pg[k] * p.page_size + sl[k]) * p.num_kv_heads + kvh) * D;
                        else
                            record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                    }
                    const uint8_t *src = (isv ? vc : kc) + (off >= 0 ? off : 0);
                    const uint32_t bytes = off >= 0 ? 16u : 0u;
                    const uint32_t drow = stg + (uint32_t)(isv * T * D + t * D);
#pragma unroll
                    for (int c = 0; c < CPR; ++c)
                        cp_async_16(drow + ((c ^ (t & SWZ)) << 4), src + c * 16, bytes);
                }
            }
            cp_async_commit();
            // The next tile, and its page ids (in flight until the next step).
            int nii = cur_ii, nj = cur_j;
            if (have && ++nj >= p.items[nii].kv_tiles) {
                nii = first_from(nii + 1);
                nj = 0;
            }
            int npg[kUPT], nsl[kUPT];
            if (nii < item_hi)
                load_ids(nii, nj, npg, nsl);
            if (staged > 0) {
                cp_async_wait<1>();
                sync_producers();  // the previous tile's rows have landed for every producer
                const uint32_t stg = sStg + (uint32_t)((staged - 1) & 1) * Tr::kStgTileBytes;
                // K, then V, each into its slot and completing that slot's barrier.
                for (int isv = 0; isv < 2; ++isv) {
                    const uint32_t pos = n + isv;
                    const int s = pos % NS;
                    const bool w_ok =
                        pos < NS || mbar_wait(bar(B::kEmpty + s), ((pos / NS) - 1) & 1, abort_v, p.wait_ns);
                    okp = bar_red_and(1, NP, w_ok);  // every producer takes the same way out
                    if (!okp)
                        break;
                    const uint32_t src0 = stg + (uint32_t)(isv * T * D), dst0 = slot(s);
                    // Consecutive threads take consecutive rows of one chunk column: the
                    // eight 16-byte accesses of a quarter warp then fall in eight
                    // different bank groups on both sides (staging and slot swizzles).
#pragma unroll 4
                    for (int u = pt; u < T * CPR; u += NP) {
                        const int t = u % T, c = u / T;
                        uint32_t w0, w1, w2, w3;
                        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                                     : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                                     : "r"(src0 + (uint32_t)(t * D) + ((c ^ (t & SWZ)) << 4))
                                     : "memory");
                        uint32_t f[8];
                        fp8x4_widen_f16<E5>(w0, f[0], f[1]);
                        fp8x4_widen_f16<E5>(w1, f[2], f[3]);
                        fp8x4_widen_f16<E5>(w2, f[4], f[5]);
                        fp8x4_widen_f16<E5>(w3, f[6], f[7]);
                        // columns 16c .. 16c+15 = granules 2(c % 4), 2(c % 4) + 1 of plane c / 4
                        const int k0 = (c & 3) * 2;
                        const uint32_t row = dst0 + (uint32_t)((c >> 2) * (T * Tr::kChunk) + t * Tr::kChunk);
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(row + ((k0 ^ (t & 7)) << 4)),
                                     "r"(f[0]), "r"(f[1]), "r"(f[2]), "r"(f[3])
                                     : "memory");
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                                         row + (((k0 + 1) ^ (t & 7)) << 4)),
                                     "r"(f[4]), "r"(f[5]), "r"(f[6]), "r"(f[7])
                                     : "memory");
                    }
                    fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
                    mbar_arrive(bar(B::kFull + s));
                }
                if (!okp)
                    break;
                n += 2;
            }
            if (!have)
                break;
            ++staged;
            cur_ii = nii;
            cur_j = nj;
#pragma unroll
            for (int k = 0; k < kUPT; ++k) {
                pg[k] = npg[k];
                sl[k] = nsl[k];
            }
        }
        if (!okp) {
            record_status(p.status, PKV_ERR_TIMEOUT);
            abort_flag = 1;
        }
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, Tr::kTmemCols);
    }
}

template <int D, int MASK, bool TMA_KV, bool RAGGED, int KV>
cudaError_t launch_pp_dmt(const PrefillParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, const CUtensorMap &to, int num_ctas, cudaStream_t s)
{
    using Tr = PPTraits<D, KV != PKV_BF16>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_pp_kernel<D, MASK, TMA_KV, RAGGED, KV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kDynSmem);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    prefill_pp_kernel<D, MASK, TMA_KV, RAGGED, KV><<<num_ctas, Tr::kThreads, Tr::kDynSmem, s>>>(p, tq, tk, tv, to);
    return cudaGetLastError();
}

template <int D, bool TMA_KV, bool RAGGED, int KV>
cudaError_t launch_pp_dt(const PrefillParams &p, int mask_mode, const CUtensorMap &tq, const CUtensorMap &tk,
                         const CUtensorMap &tv, const CUtensorMap &to, int num_ctas, cudaStream_t s)
{
    switch (mask_mode) {
    case kMaskNone: return launch_pp_dmt<D, kMaskNone, TMA_KV, RAGGED, KV>(p, tq, tk, tv, to, num_ctas, s);
    case kMaskCausal: return launch_pp_dmt<D, kMaskCausal, TMA_KV, RAGGED, KV>(p, tq, tk, tv, to, num_ctas, s);
    case kMaskCausalWindow:
        return launch_pp_dmt<D, kMaskCausalWindow, TMA_KV, RAGGED, KV>(p, tq, tk, tv, to, num_ctas, s);
    case kMaskWindow: return launch_pp_dmt<D, kMaskWindow, TMA_KV, RAGGED, KV>(p, tq, tk, tv, to, num_ctas, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pp
}  // namespace pkv
