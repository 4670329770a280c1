// Thin inline-PTX wrappers used by the kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace pkv {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy through L2 only; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// 4-byte global -> shared copy (through L1).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float m;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1) as one packed f32x2 FMA.
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                     float c1)
{
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (d0, d1) += (a0, a1) as one packed f32x2 add.
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1)
{
    asm("{\n .reg .b64 ra, rd;\n mov.b64 rd, {%0, %1};\n mov.b64 ra, {%2, %3};\n"
        " add.rn.f32x2 rd, rd, ra;\n mov.b64 {%0, %1}, rd;\n}\n"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}

// tanh from the exponential: tanh(y) = 1 - 2 / (2^(2 y log2 e) + 1), clamped to
// |y| <= 15 (tanh(15) is 1 to fp32 precision). Absolute error ~1e-7.
__device__ __forceinline__ float soft_cap_tanh(float y)
{
    y = fminf(fmaxf(y, -15.f), 15.f);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(e) : "f"(y * 2.8853900817779268f));
    return 1.f - __fdividef(2.f, e + 1.f);
}

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible (a no-op for an ordinary launch), and let
// the next grid in the stream start its own set-up.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Named barrier `id` over n threads that also ANDs a predicate across them.
__device__ __forceinline__ bool bar_red_and(int id, int n, bool pred)
{
    int r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
                 " selp.s32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((int)pred), "r"(id), "r"(n)
                 : "memory");
    return r != 0;
}

// Four 8-bit values (a 32-bit word, lowest byte first) as two f16x2 words {x0, x1},
// {x2, x3}: E4M3 through the conversion instruction, E5M2 by byte moves (an E5M2
// byte is the top byte of its f16). Every value of either format is exact in f16.
template <bool E5M2>
__device__ __forceinline__ void fp8x4_widen_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    if (E5M2) {
        lo = __byte_perm(w, 0u, 0x1404);
        hi = __byte_perm(w, 0u, 0x3424);
    } else {
        asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
            " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    }
}

__device__ __forceinline__ void record_status(int32_t *status, int32_t code)
{
    atomicCAS(status, 0, code);
}

}  // namespace pkv
