// On-device builder of kv_indptr / kv_indices from a request-to-slot table, so that
// a batch's page table can be rebuilt between CUDA-graph replays without a host
// round trip (sglang flashinfer_backend.py page, section call_begin_forward: kv_indptr
// is the running sum of the kept lengths, each request's entries are gathered from
// its row of the table starting at its kv_start, and a sliding-window pool maps them
// from full-pool locations to its own).
//
//   kv_indptr[b+1] = kv_indptr[b] + kv_lens[b]
//   kv_indices[kv_indptr[b] + j] = table[req_pool_indices[b] * row_stride + kv_start[b] + j]
//   kv_indices[i] = loc_map[kv_indices[i]]   (when a location map is given)
//
// Two launches: one CTA scans kv_lens, then one CTA per request gathers its range.
// Every read and write is bounds-checked; a violation is recorded in the optional
// status word (PKV_ERR_DEVICE_BOUNDS) and the offending entries are skipped.
#include "pkv_internal.h"
#include "pkv_nvtx.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) indptr_kernel(const int32_t *__restrict__ kv_lens, int B,
                                                              int32_t *__restrict__ indptr, int32_t *status)
{
    __shared__ int32_t warp_incl[kScanThreads / 32];
    __shared__ long long carry;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        carry = 0;
        indptr[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < B; base += kScanThreads) {
        const int i = base + threadIdx.x;
        int x = 0;
        if (i < B) {
            x = kv_lens[i];
            if (x < 0) {
                if (status)
                    record_status(status, PKV_ERR_DEVICE_BOUNDS);
                x = 0;
            }
        }
        // inclusive scan: within the warp, then over the warps' totals
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off)
                x += y;
        }
        if (lane == 31)
            warp_incl[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_incl[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off)
                    w += y;
            }
            warp_incl[lane] = w;
        }
        __syncthreads();
        const long long incl = carry + x + (warp > 0 ? warp_incl[warp - 1] : 0);
        if (i < B) {
            if (incl > 0x7fffffffLL && status)
                record_status(status, PKV_ERR_DEVICE_BOUNDS);
            indptr[i + 1] = (int32_t)incl;
        }
        __syncthreads();  // every thread has read carry
        if (threadIdx.x == kScanThreads - 1)
            carry = incl;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) gather_kernel(const int32_t *__restrict__ table, int32_t num_rows,
                                                     int64_t row_stride, const int32_t *__restrict__ req_pool_indices,
                                                     const int32_t *__restrict__ kv_start,
                                                     const int32_t *__restrict__ kv_lens,
                                                     const int32_t *__restrict__ indptr,
                                                     const int32_t *__restrict__ loc_map, int64_t loc_map_len,
                                                     int32_t *__restrict__ out, int64_t capacity, int32_t *status)
{
    const int b = blockIdx.x;
    const int len = kv_lens[b];
    if (len <= 0)
        return;
    const int row = req_pool_indices[b];
    const int start = kv_start[b];
    const long long o = indptr[b];
    if (row < 0 || row >= num_rows || start < 0 || (long long)start + len > row_stride || o < 0 ||
        o + len > capacity) {
        if (threadIdx.x == 0 && status)
            record_status(status, PKV_ERR_DEVICE_BOUNDS);
        return;
    }
    const int32_t *src = table + (long long)row * row_stride + start;
    for (int j = threadIdx.x; j < len; j += blockDim.x) {
        int32_t x = src[j];
        if (loc_map) {
            if ((unsigned long long)(long long)x < (unsigned long long)loc_map_len) {
                x = loc_map[x];
            } else {
                if (status)
                    record_status(status, PKV_ERR_DEVICE_BOUNDS);
                x = -1;  // an invalid page id: attention kernels record it too
            }
        }
        out[o + j] = x;
    }
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int pkv_build_kv_indices(const int32_t *req_to_token, int32_t num_rows, int64_t row_stride,
                                            const int32_t *req_pool_indices, const int32_t *kv_start,
                                            const int32_t *kv_lens, int32_t batch_size, const int32_t *loc_map,
                                            int64_t loc_map_len, int32_t *kv_indptr, int32_t *kv_indices,
                                            int64_t kv_indices_capacity, int32_t *status, void *stream_)
{
    using namespace pkv;
    NvtxRange range("pkv_build_kv_indices");
    if (batch_size < 0 || num_rows < 0 || row_stride < 0 || kv_indices_capacity < 0 || loc_map_len < 0) {
        set_last_error("pkv_build_kv_indices: negative size");
        return PKV_ERR_INVALID_ARG;
    }
    if (!kv_indptr || (batch_size > 0 && (!req_to_token || !req_pool_indices || !kv_start || !kv_lens)) ||
        (kv_indices_capacity > 0 && !kv_indices)) {
        set_last_error("pkv_build_kv_indices: a required pointer is NULL");
        return PKV_ERR_INVALID_ARG;
    }
    if (loc_map && loc_map_len == 0) {
        set_last_error("pkv_build_kv_indices: loc_map given with loc_map_len 0");
        return PKV_ERR_INVALID_ARG;
    }
    cudaStream_t stream = (cudaStream_t)stream_;
    indptr_kernel<<<1, kScanThreads, 0, stream>>>(kv_lens, batch_size, kv_indptr, status);
    cudaError_t ce = cudaGetLastError();
    if (ce == cudaSuccess && batch_size > 0) {
        gather_kernel<<<batch_size, 256, 0, stream>>>(req_to_token, num_rows, row_stride, req_pool_indices, kv_start,
                                                      kv_lens, kv_indptr, loc_map, loc_map_len, kv_indices,
                                                      kv_indices_capacity, status);
        ce = cudaGetLastError();
    }
    if (ce != cudaSuccess) {
        set_last_error(cudaGetErrorString(ce));
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}
