// scan_util.cuh -- device helpers shared by the compute_out kernels (k_chunk_scan.cu,
// k_chunk_scan_pair.cu): bounded role waits, packing to 16-bit pairs, 32-byte global
// accesses and the in-sub-block log2 decay.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "sm100.cuh"

namespace ssd {

// The roles' waits.  INL: the whole loop inlined at every site (no call, so no register save and
// restore through local memory around it), measured 3-4% faster for the plain kernel; the larger
// instantiation with the layer's output options measured faster with the shared out-of-line loop.
template <bool INL>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, int code,
                                             uint64_t limit_ns) {
    if constexpr (INL) return sm100::mbar_wait_bounded_inline(bar, parity, abort, err, code, limit_ns);
    else return sm100::mbar_wait_bounded(bar, parity, abort, err, code, limit_ns);
}

// 32 bytes from a 32-byte-aligned read-only global address in one load (sm_100+ 256-bit vector load)
__device__ __forceinline__ void ld_global_nc_32B(const void* p, uint4& lo, uint4& hi) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
                 : "l"(p));
}

// a thread's 128-byte z row: 32-byte loads when z is 32-byte aligned, else 16-byte loads
__device__ __forceinline__ void load_z_row(const uint4* zr, bool z32, uint4 (&zq)[8]) {
    if (z32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_global_nc_32B(zr + 2 * i, zq[2 * i], zq[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) zq[i] = __ldg(zr + i);
    }
}

// 32 bytes to a 32-byte-aligned global address in one store (sm_100+ 256-bit vector store)
__device__ __forceinline__ void st_global_32B(void* p, const uint4& lo, const uint4& hi) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(lo.x), "r"(lo.y), "r"(lo.z),
                 "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// In-sub-block inclusive log2 decay of position i (raw per-chunk cumsums in
// scs, the raw value before the sub-block in prev when it starts inside a
// chunk; a 64-token chunk boundary may fall inside the sub-block).
__device__ __forceinline__ float sub_block_decay(const float* scs, float prev, int p0, int Q, int i) {
    return ((p0 + i) / Q == 0) ? (scs[i] - prev) : ((scs[Q - 1 - p0] - prev) + scs[i]);
}

// |packed float16 pair| folded into a running maximum: a value that rounded past 65504 became an
// infinity, so the maximum exceeds float16's range exactly when some converted value did
__device__ __forceinline__ void hmax_abs(__half2& acc, uint32_t packed) {
    __half2 v = *reinterpret_cast<const __half2*>(&packed);
    acc = __hmax2(acc, __habs2(v));
}

// Four packed pairs folded at once, as a tree: a chain of one dependent maximum per four pairs.
__device__ __forceinline__ void hmax_abs4(__half2& acc, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    const __half2 ab = __hmax2(__habs2(*reinterpret_cast<const __half2*>(&a)), __habs2(*reinterpret_cast<const __half2*>(&b)));
    const __half2 cd = __hmax2(__habs2(*reinterpret_cast<const __half2*>(&c)), __habs2(*reinterpret_cast<const __half2*>(&d)));
    acc = __hmax2(acc, __hmax2(ab, cd));
}

// Two float32 products in one instruction (sm_100's packed two-lane multiply, round to nearest even,
// the same result as two separate multiplies).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Two float32 fused multiply-adds a * b + c in one instruction (round to nearest even per lane).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float hmax_to_float(__half2 acc) {
    return fmaxf(__low2float(acc), __high2float(acc));
}

}  // namespace ssd
