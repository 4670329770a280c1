// LSE merge kernels.
//
// merge_state (sglang flashinfer_backend.py page, sections _safe_merge_state and
// forward_extend, where the ragged extend partial meets the paged prefix partial): for two states over
// disjoint key sets, s = ln(e^s_a + e^s_b) and v = (e^s_a v_a + e^s_b v_b) / e^s.
// The split-KV pass generalises it to n partial states of one row.
//
// One warp per (token, head) row, D/32 contiguous elements per lane (vectorised
// 8- to 32-byte accesses); the grid is a flat range of rows, so the head count
// has no per-block limit (the pages fall back to another kernel when
// head_dim / vec_size x num_heads exceeds 1024 threads per block).
#include <cfloat>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int N>
__device__ __forceinline__ void load_vals(const float *src, float (&x)[N])
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src + i);
            x[i] = t.x; x[i + 1] = t.y; x[i + 2] = t.z; x[i + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float2 t = *reinterpret_cast<const float2 *>(src + i);
            x[i] = t.x; x[i + 1] = t.y;
        }
    }
}

template <int N>
__device__ __forceinline__ void load_vals(const uint16_t *src, float (&x)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(src + i);
        x[i] = __uint_as_float(w << 16);
        x[i + 1] = __uint_as_float(w & 0xffff0000u);
    }
}

template <int N>
__device__ __forceinline__ void store_vals(float *dst, const float (&x)[N])
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4)
            *reinterpret_cast<float4 *>(dst + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 2)
            *reinterpret_cast<float2 *>(dst + i) = make_float2(x[i], x[i + 1]);
    }
}

template <int N>
__device__ __forceinline__ void store_vals(uint16_t *dst, const float (&x)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 2)
        *reinterpret_cast<uint32_t *>(dst + i) = pack_bf16(x[i], x[i + 1]);
}

template <int D, typename V>
__global__ void __launch_bounds__(256) merge_state_kernel(const V *v_a, const float *s_a, const V *v_b,
                                                          const float *s_b, V *v_out, float *s_out,
                                                          int64_t rows)
{
    constexpr int N = D / 32;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    const float sa = s_a[row], sb = s_b[row];
    const float mx = fmaxf(sa, sb);
    float xa[N], xb[N], y[N];
    load_vals<N>(v_a + row * D + lane * N, xa);
    load_vals<N>(v_b + row * D + lane * N, xb);
    float s;
    if (mx == -INFINITY) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            y[i] = 0.f;
        s = -INFINITY;
    } else {
        const float wa = fast_exp2((sa - mx) * kLog2e);
        const float wb = fast_exp2((sb - mx) * kLog2e);
        const float inv = 1.f / (wa + wb);
        const float fa = wa * inv, fb = wb * inv;
#pragma unroll
        for (int i = 0; i < N; ++i)
            y[i] = fa * xa[i] + fb * xb[i];
        s = mx + __log2f(wa + wb) * kLn2;
    }
    __syncwarp();  // v_out may alias v_a: every lane has read before anyone writes
    store_vals<N>(v_out + row * D + lane * N, y);
    if (lane == 0)
        s_out[row] = s;
}

template <int D>
__global__ void __launch_bounds__(256) merge_partials_kernel(const MergePartialsParams p)
{
    constexpr int N = D / 32;
    const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= (int64_t)p.num_items * p.num_qo_heads)
        return;
    const MergeItem it = p.items[gw / p.num_qo_heads];
    const int h = (int)(gw % p.num_qo_heads);
    float mx = -INFINITY;
    for (int k = lane; k < it.num_partials; k += 32)
        mx = fmaxf(mx, p.partial_lse[(size_t)(it.partial_begin + k) * p.num_qo_heads + h]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float acc[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        acc[i] = 0.f;
    float sum = 0.f;
    if (mx != -INFINITY) {
        for (int k = 0; k < it.num_partials; ++k) {
            const size_t slot = (size_t)(it.partial_begin + k) * p.num_qo_heads + h;
            const float w = fast_exp2((p.partial_lse[slot] - mx) * kLog2e);
            float x[N];
            load_vals<N>(p.partial_o + slot * D + lane * N, x);
#pragma unroll
            for (int i = 0; i < N; ++i)
                acc[i] += w * x[i];
            sum += w;
        }
    }
    const float inv = sum > 0.f ? p.v_scale / sum : 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        acc[i] *= inv;
    store_vals<N>(p.out + ((size_t)it.row * p.num_qo_heads + h) * D + lane * N, acc);
    if (lane == 0 && p.lse)
        p.lse[(size_t)it.row * p.num_qo_heads + h] = sum > 0.f ? mx + __log2f(sum) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t merge_state_d(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                          void *v_out, float *s_out, int64_t rows, int dtype, cudaStream_t s)
{
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (dtype == PKV_F32)
        merge_state_kernel<D, float><<<grid, 256, 0, s>>>((const float *)v_a, s_a, (const float *)v_b,
                                                          s_b, (float *)v_out, s_out, rows);
    else
        merge_state_kernel<D, uint16_t><<<grid, 256, 0, s>>>((const uint16_t *)v_a, s_a,
                                                             (const uint16_t *)v_b, s_b,
                                                             (uint16_t *)v_out, s_out, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_state(const void *v_a, const float *s_a, const void *v_b, const float *s_b,
                               void *v_out, float *s_out, int64_t rows, int head_dim, int dtype,
                               cudaStream_t s)
{
    if ((rows + 7) / 8 > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    switch (head_dim) {
    case 64: return merge_state_d<64>(v_a, s_a, v_b, s_b, v_out, s_out, rows, dtype, s);
    case 128: return merge_state_d<128>(v_a, s_a, v_b, s_b, v_out, s_out, rows, dtype, s);
    case 256: return merge_state_d<256>(v_a, s_a, v_b, s_b, v_out, s_out, rows, dtype, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_merge_partials(const MergePartialsParams &p, int head_dim, cudaStream_t s)
{
    const int64_t warps = (int64_t)p.num_items * p.num_qo_heads;
    const unsigned grid = (unsigned)((warps + 7) / 8);
    switch (head_dim) {
    case 64: merge_partials_kernel<64><<<grid, 256, 0, s>>>(p); break;
    case 128: merge_partials_kernel<128><<<grid, 256, 0, s>>>(p); break;
    case 256: merge_partials_kernel<256><<<grid, 256, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pkv
