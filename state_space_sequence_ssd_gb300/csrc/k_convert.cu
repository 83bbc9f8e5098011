// k_convert.cu -- bfloat16 -> float16 copy of the B and C inputs.
//
// The tensor-core products whose operands are derived values (the masked
// decay matrix, the carried state, the decay-scaled x rows) need more than
// bfloat16's 8 significant bits to meet the output tolerance, and a tcgen05
// kind::f16 MMA takes both operands in one type.  float16 carries 11
// significant bits, and every bfloat16 value with magnitude in
// [2^-14, 65504] converts to float16 exactly, so the kernels run all four
// products in float16 on exact copies of the inputs.  Magnitudes above 65504
// saturate to +-65504 and raise the library's float16 range flag (the call
// then reports SSD_ERR_RANGE); below 2^-14 they keep float16's subnormal
// precision.
#include <cuda_fp16.h>

#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// two bfloat16 -> two float16 (saturating); mx tracks the largest magnitude seen
__device__ __forceinline__ uint32_t cvt_pair(uint32_t v, float& mx) {
    const float lo = __uint_as_float(v << 16);
    const float hi = __uint_as_float(v & 0xffff0000u);
    mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
    const __half2 h = __floats2half2_rn(fminf(fmaxf(lo, -kF16Max), kF16Max), fminf(fmaxf(hi, -kF16Max), kF16Max));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// converts a[0..n16) and, if b is given, b[0..n16) (16-byte chunks of 8 values)
__global__ void __launch_bounds__(kThreads) bf16_to_f16_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b,
                                                               uint4* __restrict__ oa, uint4* __restrict__ ob,
                                                               int64_t n16, int* err) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t total = (b != nullptr) ? 2 * n16 : n16;
    float mx = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += stride) {
        const bool second = i >= n16;
        const int64_t j = second ? i - n16 : i;
        uint4 v = second ? b[j] : a[j];
        v.x = cvt_pair(v.x, mx);
        v.y = cvt_pair(v.y, mx);
        v.z = cvt_pair(v.z, mx);
        v.w = cvt_pair(v.w, mx);
        (second ? ob : oa)[j] = v;
    }
    flag_f16_range(err, mx);
}

}  // namespace

int launch_bc_to_f16(const __nv_bfloat16* B, const __nv_bfloat16* C, const Dims& d, __half* B16, __half* C16,
                     int* err, cudaStream_t s) {
    const int64_t n = (int64_t)d.batch * d.seqlen * d.ngroups * d.dstate;  // multiple of 64
    const int64_t n16 = n / 8;
    int64_t blocks = ((C != nullptr ? 2 : 1) * n16 + kThreads - 1) / kThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    launch_begin(kKindConvert, s);
    bf16_to_f16_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(B),
                                                               reinterpret_cast<const uint4*>(C),
                                                               reinterpret_cast<uint4*>(B16),
                                                               reinterpret_cast<uint4*>(C16), n16, err);
    return launch_end(kKindConvert, s);
}

}  // namespace ssd
