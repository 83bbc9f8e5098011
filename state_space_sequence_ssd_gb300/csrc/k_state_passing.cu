// k_state_passing.cu -- second half of fwd_pass_state: the sequential hop
// across chunks.
//
// devotd.net page on the Mamba-2 cuTile forward kernels, section 2
// (fwd_pass_state keeps chunk order but processes independent parts of the
// state in parallel); disconfirmai.com page "Jane Street ML Engineers Map
// Mamba-2 Recurrent State Computation to Tensor Cores with cuTile",
// jump-formula paragraph (the decay re-enters as an exponential of the
// log-space chunk sum).
//
//   h_0 = init;  states[c] = h_c;  h_{c+1} = 2^(cs[b,h,c,Q-1]) h_c + S[c];  final = h_nc
//
// Reverse mode (the backward pass): the steps run from the last chunk to the
// first, so with the gradient into the final state as `init` the hop gives,
// per chunk, the gradient flowing into the state after it from later tokens,
// and as `final` the gradient with respect to the initial state:
//   mu_{nc-1} = dfinal;  out[c] = mu_c;  mu_{c-1} = 2^(cs[b,h,c,Q-1]) mu_c + Z[c];  final = mu_{-1}
//
// With `states16` given, the per-step states are written as float16 there
// instead (the backward pass, whose kernel reads them as tensor-core operands);
// a value past float16's range raises the range flag of `err`.  With `S16`
// given, the per-step terms are read as float16 from there (the backward
// pass's per-block terms; the recurrence itself stays float32).
//
// Every (b, h, p, n) entry is an independent lane of a serial fp32 recurrence.
// Each thread owns 4 consecutive entries (one float4); the loop over chunks
// keeps two groups of U chunk-state loads in flight -- the next group is
// requested before the current one is folded -- so the memory system always
// has independent requests outstanding (the loads of S do not depend on the
// carried state).  U = 8 for float32 terms and 16 for float16 ones, so that
// a thread keeps the same bytes in flight.  `states` may alias `S`: every element is
// read before the same element is written.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// four consecutive per-step terms as loaded: float32, or float16 (H16) kept packed until they are folded
template <bool H16>
struct Term {
    using T = float4;
    static __device__ __forceinline__ T load(const float* S, const __half*, int64_t i) {
        return *reinterpret_cast<const float4*>(S + i);
    }
    static __device__ __forceinline__ float4 widen(const T& v) { return v; }
};
template <>
struct Term<true> {
    using T = uint2;
    static __device__ __forceinline__ T load(const float*, const __half* S16, int64_t i) {
        return *reinterpret_cast<const uint2*>(S16 + i);
    }
    static __device__ __forceinline__ float4 widen(const T& u) {
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
};

// dec: log2 decay of step c for row (b, h) at dec[row * dec_row + c * dec_step]
template <bool H16>
__global__ void __launch_bounds__(kThreads) state_passing_kernel(const float* S, const __half* S16,
                                                                 const float* __restrict__ dec,
                                                                 int64_t dec_step, int64_t dec_row,
                                                                 const float* __restrict__ init, Dims d,
                                                                 float* states, float* __restrict__ final_state,
                                                                 int rev, __half* states16, int* err) {
    grid_dep_wait();  // the chunk or span states come from the previous launch
    grid_dep_launch_dependents();
    const int64_t PN = (int64_t)d.headdim * d.dstate;
    const int64_t e = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * 4;
    const int h = blockIdx.y, b = blockIdx.z;
    if (e >= PN) return;
    const int nc = d.nchunks;
    float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
    // h: local head (S, states and dec hold the call's hcount heads); init and final are caller tensors
    // indexed by the global head head0 + h
    if (init != nullptr) hv = *reinterpret_cast<const float4*>(init + ((int64_t)b * d.nheads + d.head0 + h) * PN + e);
    const float* csl = dec + ((int64_t)b * d.hcount + h) * dec_row;
    const int64_t cstride = (int64_t)d.hcount * PN;  // distance between consecutive chunks
    const int64_t base = ((int64_t)b * nc * d.hcount + h) * PN + e;
    // software pipeline: the next group of kUnroll steps is loaded before the current one is folded
    constexpr int kUnroll = H16 ? 16 : 8;
    float mx = 0.f;  // largest |state| written as float16
    typename Term<H16>::T sv[kUnroll], nv[kUnroll];
    float dk[kUnroll], nd[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
        if (k < nc) {
            const int c = rev ? nc - 1 - k : k;
            nv[k] = Term<H16>::load(S, S16, base + (int64_t)c * cstride);
            nd[k] = __ldg(csl + (int64_t)c * dec_step);
        }
    }
    for (int c0 = 0; c0 < nc; c0 += kUnroll) {
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            sv[k] = nv[k];
            dk[k] = nd[k];
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int cn = c0 + kUnroll + k;
            if (cn < nc) {
                const int c = rev ? nc - 1 - cn : cn;
                nv[k] = Term<H16>::load(S, S16, base + (int64_t)c * cstride);
                nd[k] = __ldg(csl + (int64_t)c * dec_step);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            if (c0 + k < nc) {
                const float dd = exp2f(dk[k]);
                const int c = rev ? nc - 1 - (c0 + k) : c0 + k;
                if (states16 != nullptr) {
                    const __half2 lo = __floats2half2_rn(hv.x, hv.y), hi = __floats2half2_rn(hv.z, hv.w);
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(hv.x), fabsf(hv.y)), fmaxf(fabsf(hv.z), fabsf(hv.w))));
                    uint2 o16;
                    o16.x = *reinterpret_cast<const uint32_t*>(&lo);
                    o16.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(states16 + base + (int64_t)c * cstride) = o16;
                } else {
                    *reinterpret_cast<float4*>(states + base + (int64_t)c * cstride) = hv;
                }
                const float4 tv = Term<H16>::widen(sv[k]);
                hv.x = fmaf(dd, hv.x, tv.x);
                hv.y = fmaf(dd, hv.y, tv.y);
                hv.z = fmaf(dd, hv.z, tv.z);
                hv.w = fmaf(dd, hv.w, tv.w);
            }
        }
    }
    if (final_state != nullptr)
        *reinterpret_cast<float4*>(final_state + ((int64_t)b * d.nheads + d.head0 + h) * PN + e) = hv;
    if (!(mx <= kF16Max) && err != nullptr) atomicOr(err + 1, 1);  // a float16 state out of range
}

}  // namespace

int launch_state_passing(const float* S, const float* cs, const float* init, const Dims& d,
                         float* states, float* final_state, cudaStream_t s) {
    // per-chunk decay: cs[b, h, c, Q-1]
    return launch_state_passing_steps(S, cs + (d.chunk_size - 1), d.chunk_size, (int64_t)d.nchunks * d.chunk_size,
                                      init, d, d.nchunks, states, final_state, s);
}

int launch_state_passing_steps(const float* S, const float* dec, int64_t dec_step, int64_t dec_row,
                               const float* init, const Dims& d, int nsteps, float* states, float* final_state,
                               cudaStream_t s, int rev, __half* states16, int* err, const __half* S16) {
    Dims dd = d;
    dd.nchunks = nsteps;
    const int64_t PN = (int64_t)d.headdim * d.dstate;
    dim3 grid((unsigned)ceil_div64(PN, (int64_t)kThreads * 4), d.hcount, d.batch);
    launch_begin(kKindStatePassing, s);
    const cudaError_t le =
        S16 != nullptr
            ? launch_dependent(state_passing_kernel<true>, grid, dim3(kThreads), 0, s, S, S16, dec, dec_step, dec_row,
                               init, dd, states, final_state, rev, states16, err)
            : launch_dependent(state_passing_kernel<false>, grid, dim3(kThreads), 0, s, S, S16, dec, dec_step, dec_row,
                               init, dd, states, final_state, rev, states16, err);
    const int r = launch_end(kKindStatePassing, s);
    return le != cudaSuccess ? SSD_ERR_CUDA : r;
}

}  // namespace ssd
