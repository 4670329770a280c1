// Split-KV paged decode kernel: one query row per request, the whole query-head
// group of a KV head against each streamed K/V row (GQA packing, flashinfer_backend.py
// should_use_tensor_core: the head group is fused into the MMA rows), online softmax
// in fp32, fp32 partial states per split for the merge pass.
//
// The plan has already clipped each CTA's key range [j0, j1) to the visible
// interval [p - W, p] of the request's single query position, so inside the range
// every key is visible; the kernel only masks the padding past j1 in its last tile.
//
// Data path per CTA (4 warps, 128 threads):
//   cp.async 16-byte gathers of K and V rows, one page-table lookup per row, into
//   a 3-stage ring of XOR-swizzled shared-memory tiles of 64 tokens;
//   warp w takes tokens [16w, 16w + 16) of each tile: S = Q K^T and O += P V with
//   mma.sync m16n8k16 (bf16 in, fp32 accumulate), rows = the query heads (<= 16);
//   the four warps keep independent (m, l, O) and are merged once at the end.
#include <cfloat>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

template <int D>
struct DecodeTraits {
    static constexpr int kTile = 64;  // KV tokens per pipeline stage
    static constexpr int kThreads = 128;
    static constexpr int kChunks = D / 8;  // 16-byte chunks per row
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kTile * kRowBytes;  // K or V of one stage
    static constexpr int kStages = 3;
    static constexpr int kQBytes = kDecodeRows * kRowBytes;
    static constexpr int kPipeBytes = kStages * 2 * kTileBytes;
    static constexpr int kORowFloats = D + 8;  // padded row of the combine buffer
    static constexpr int kCombineBytes = 4 * kDecodeRows * kORowFloats * 4;
    static constexpr int kSmem =
        kQBytes + (kPipeBytes > kCombineBytes ? kPipeBytes : kCombineBytes);
    static constexpr int kMinBlocks = D >= 256 ? 1 : 2;
};

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile with D-wide rows;
// chunks are XOR-swizzled by row so that ldmatrix of 8 rows hits 8 bank groups.
template <int D>
__device__ __forceinline__ int swz(int row, int chunk)
{
    return row * (D * 2) + ((chunk ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(128, DecodeTraits<D>::kMinBlocks)
    decode_kernel(const DecodeParams p)
{
    using T = DecodeTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ float red_m[4][kDecodeRows];
    __shared__ float red_l[4][kDecodeRows];
    __shared__ float row_m[kDecodeRows];
    __shared__ float row_inv_l[kDecodeRows];

    uint8_t *sQ = smem;
    uint8_t *sKV = smem + T::kQBytes;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const DecodeItem it = p.items[blockIdx.x];
    const RequestInfo rq = p.reqs[it.req];
    const int n = it.j1 - it.j0;
    const int ntiles = n > 0 ? (n + T::kTile - 1) / T::kTile : 0;

    // Q rows: query heads head0 .. head0 + nheads - 1 of the request's row; the rest zero.
    for (int idx = tid; idx < kDecodeRows * T::kChunks; idx += T::kThreads) {
        const int r = idx / T::kChunks, c = idx % T::kChunks;
        const int h = it.head0 + (r < it.nheads ? r : 0);
        const uint16_t *src = p.q + ((size_t)rq.qo_begin * p.num_qo_heads + h) * D + c * 8;
        cp_async_16(smem_u32(sQ + swz<D>(r, c)), src, r < it.nheads ? 16u : 0u);
    }
    cp_async_commit();

    auto load_tile = [&](int t, int stage) {
        uint8_t *sK = sKV + stage * 2 * T::kTileBytes;
        uint8_t *sV = sK + T::kTileBytes;
        constexpr int kRowsPerPass = T::kThreads / T::kChunks;
        const int c = tid % T::kChunks;
#pragma unroll
        for (int r0 = 0; r0 < T::kTile; r0 += kRowsPerPass) {
            const int r = r0 + tid / T::kChunks;
            const int j = it.j0 + t * T::kTile + r;
            const uint16_t *ks = p.k_cache;
            const uint16_t *vs = p.v_cache;
            uint32_t bytes = 0;
            if (j < it.j1) {
                const int lp = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                const int slot = j - lp * p.page_size;
                const int page = __ldg(p.kv_indices + rq.kv_page_begin + lp);
                if ((unsigned)page < (unsigned)p.num_pages) {
                    const size_t off =
                        (((size_t)page * p.page_size + slot) * p.num_kv_heads + it.kv_head) * D + c * 8;
                    ks += off;
                    vs += off;
                    bytes = 16;
                } else {
                    record_status(p.status, PKV_ERR_DEVICE_BOUNDS);
                }
            }
            cp_async_16(smem_u32(sK + swz<D>(r, c)), ks, bytes);
            cp_async_16(smem_u32(sV + swz<D>(r, c)), vs, bytes);
        }
    };

#pragma unroll
    for (int s = 0; s < T::kStages - 1; ++s) {
        if (s < ntiles)
            load_tile(s, s);
        cp_async_commit();
    }

    cp_async_wait<T::kStages - 1>();  // the Q group has landed
    __syncthreads();
    uint32_t qf[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int mi = lane >> 3;
        const int row = ((mi & 1) << 3) + (lane & 7);
        const int ch = 2 * ks + (mi >> 1);
        ldmatrix_x4(smem_u32(sQ + swz<D>(row, ch)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }

    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const float scale = p.sm_scale_log2;

    for (int t = 0; t < ntiles; ++t) {
        const int stage = t % T::kStages;
        cp_async_wait<T::kStages - 2>();
        __syncthreads();
        {
            const int tn = t + T::kStages - 1;
            if (tn < ntiles)
                load_tile(tn, tn % T::kStages);
            cp_async_commit();
        }
        const uint8_t *sK = sKV + stage * 2 * T::kTileBytes;
        const uint8_t *sV = sK + T::kTileBytes;

        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int mi = lane >> 3;
            const int row = warp * 16 + ((mi >> 1) << 3) + (lane & 7);
            const int ch = 2 * ks + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(smem_u32(sK + swz<D>(row, ch)), b0, b1, b2, b3);
            mma_bf16_16816(s[0], qf[ks], b0, b1);
            mma_bf16_16816(s[1], qf[ks], b2, b3);
        }
        const int tok_base = t * T::kTile + warp * 16 + 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = tok_base + nt * 8 + (e & 1);
                s[nt][e] = tok < n ? s[nt][e] * scale : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
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
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = fast_exp2(s[nt][0] - ref0);
            pr[nt][1] = fast_exp2(s[nt][1] - ref0);
            pr[nt][2] = fast_exp2(s[nt][2] - ref1);
            pr[nt][3] = fast_exp2(s[nt][3] - ref1);
        }
        l[0] = l[0] * a0 + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
        l[1] = l[1] * a1 + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= a0;
            o[i][1] *= a0;
            o[i][2] *= a1;
            o[i][3] *= a1;
        }
        const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                                pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
            const int mi = lane >> 3;
            const int row = warp * 16 + ((mi & 1) << 3) + (lane & 7);
            const int ch = 2 * np + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(smem_u32(sV + swz<D>(row, ch)), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * np], pa, b0, b1);
            mma_bf16_16816(o[2 * np + 1], pa, b2, b3);
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // the ring is free for the combine buffer

    // Merge the four warps' states.
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
    __syncthreads();
    if (tid < kDecodeRows) {
        float M = fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]), fmaxf(red_m[2][tid], red_m[3][tid]));
        const float ref = M == -INFINITY ? 0.f : M;
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            L += red_l[w][tid] * fast_exp2(red_m[w][tid] - ref);
        row_m[tid] = M;
        row_inv_l[tid] = L > 0.f ? 1.f / L : 0.f;
        if (tid < it.nheads) {
            const float lse_v = L > 0.f ? (M + __log2f(L)) * 0.6931471805599453f : -INFINITY;
            const int h = it.head0 + tid;
            if (it.partial >= 0)
                p.partial_lse[(size_t)it.partial * p.num_qo_heads + h] = lse_v;
            else if (p.lse)
                p.lse[(size_t)rq.qo_begin * p.num_qo_heads + h] = lse_v;
        }
    }
    __syncthreads();
    float *sO = reinterpret_cast<float *>(sKV);
    {
        const float M0 = row_m[r0], M1 = row_m[r1];
        const float f0 = fast_exp2(m[0] - (M0 == -INFINITY ? 0.f : M0)) * row_inv_l[r0];
        const float f1 = fast_exp2(m[1] - (M1 == -INFINITY ? 0.f : M1)) * row_inv_l[r1];
        float *w0 = sO + (warp * kDecodeRows + r0) * T::kORowFloats + 2 * (lane & 3);
        float *w1 = sO + (warp * kDecodeRows + r1) * T::kORowFloats + 2 * (lane & 3);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            *reinterpret_cast<float2 *>(w0 + 8 * i) = make_float2(o[i][0] * f0, o[i][1] * f0);
            *reinterpret_cast<float2 *>(w1 + 8 * i) = make_float2(o[i][2] * f1, o[i][3] * f1);
        }
    }
    __syncthreads();
    for (int idx = tid; idx < kDecodeRows * (D / 8); idx += T::kThreads) {
        const int r = idx / (D / 8);
        const int c = (idx % (D / 8)) * 8;
        if (r >= it.nheads)
            continue;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[e] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float4 *src = reinterpret_cast<const float4 *>(sO + (w * kDecodeRows + r) * T::kORowFloats + c);
            const float4 x = src[0], y = src[1];
            acc[0] += x.x; acc[1] += x.y; acc[2] += x.z; acc[3] += x.w;
            acc[4] += y.x; acc[5] += y.y; acc[6] += y.z; acc[7] += y.w;
        }
        const int h = it.head0 + r;
        if (it.partial >= 0) {
            float4 *dst = reinterpret_cast<float4 *>(p.partial_o + ((size_t)it.partial * p.num_qo_heads + h) * D + c);
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

template <int D>
cudaError_t launch_decode_d(const DecodeParams &p, int num_items, cudaStream_t s)
{
    using T = DecodeTraits<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             T::kSmem);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    decode_kernel<D><<<num_items, T::kThreads, T::kSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int head_dim, int num_items, cudaStream_t s)
{
    switch (head_dim) {
    case 64: return launch_decode_d<64>(p, num_items, s);
    case 128: return launch_decode_d<128>(p, num_items, s);
    case 256: return launch_decode_d<256>(p, num_items, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
