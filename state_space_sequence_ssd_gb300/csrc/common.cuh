// common.cuh -- shared host/device definitions of the SSD library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

constexpr float kLog2e = 1.4426950408889634f;

// Per-launch failure handling of the pipelined tensor-core kernels.
//   err[0]   code of the first bounded wait that gave up (0: none) -- reported as SSD_ERR_TIMEOUT;
//   err[1]   non-zero once a value converted to a float16 tensor-core operand fell outside
//            float16's finite range (|v| > 65504) -- reported as SSD_ERR_RANGE.
//   wait_ns  limit of every pipeline wait (drains at teardown use kDrainNs instead);
//   stall    test hook: the kernel first waits on a barrier that nothing completes, so that the
//            wait runs out and the abort path runs (see ssd_debug_stall in ssd.h).
struct Ctl {
    int* err = nullptr;
    unsigned long long wait_ns = 1000000000ull;
    int stall = 0;
};

// Limit of the teardown drains (copies and products already issued always complete).
constexpr unsigned long long kDrainNs = 1000000000ull;

// Largest finite float16 magnitude.
constexpr float kF16Max = 65504.f;

// Called by all 32 lanes of a warp: raises the float16 range flag if any lane saw a value whose
// magnitude `mx` (the largest it converted to float16, or NaN) is not finite in float16.
__device__ __forceinline__ void flag_f16_range(int* err, float mx) {
    const bool bad = !(mx <= kF16Max);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && err != nullptr) atomicOr(err + 1, 1);
}

// Problem dimensions shared by every launch.  A call may cover a contiguous range of heads of
// full-size tensors: heads head0 .. head0 + hcount - 1 of nheads.  Caller tensors (x, y, dt, A, D, z,
// init and final states) are indexed by the global head h = head0 + local head; the library's own
// intermediates (dA_cumsum and dt rows, chunk or span states and decays) hold the hcount heads of the
// call only and are indexed by the local head.  A whole-problem call has head0 = 0, hcount = nheads.
struct Dims {
    int batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, nchunks;
    int head0, hcount;
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The dt transform of the input-side options (ssd_input_options): bias, then
// softplus, then clamp; identity when nothing is set.
struct DtOpts {
    const float* bias = nullptr;  // (H) or nullptr
    int softplus = 0;
    int limit = 0;
    float lo = 0.f, hi = 0.f;
    __host__ __device__ bool active() const { return bias != nullptr || softplus != 0 || limit != 0; }
};

// log(1 + exp(v)) written as max(v, 0) + log(1 + exp(-|v|)), which never overflows.
__device__ __forceinline__ float effective_dt(float v, int h, const DtOpts& o) {
    if (o.bias != nullptr) v += __ldg(o.bias + h);
    if (o.softplus) v = fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
    if (o.limit) v = fminf(fmaxf(v, o.lo), o.hi);
    return v;
}

// Output-side options: one skip weight per channel (D is (H, P)) and the z gate.
struct OutOpts {
    const float* Dp = nullptr;            // (H, P) or nullptr
    const __nv_bfloat16* z = nullptr;     // x's layout or nullptr
};

// z sigmoid(z) = z / (1 + exp(-z)), with the approximate division: for z < -87 the
// denominator exceeds 2^126 and the quotient is 0, the function's limit.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Programmatic dependent launch.  A kernel launched with launch_dependent() may begin while
// the previous kernel on the stream is still running; it must execute grid_dep_wait() before
// it reads anything an earlier launch wrote (the wait returns once that kernel has completed
// and its writes are visible).  grid_dep_launch_dependents() lets the next such launch begin.
// Both are no-ops for a kernel launched without the attribute or followed by none.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Kernel kinds, for the profiling counters (names in ssd_api.cu).
enum KernelKind {
    kKindCumsum = 0,
    kKindChunkState = 1,
    kKindStatePassing = 2,
    kKindChunkScan = 3,
    kKindConvert = 4,
    kKindStep = 5,
    kKindBwdChunk = 6,
    kKindBwdReduce = 7,
    kNumKinds = 8
};

// Sets a kernel's dynamic shared-memory limit once per (kernel, device).
int ensure_smem_limit(const void* kernel, int bytes);

// Launch bookkeeping implemented in ssd_api.cu: opens/closes the optional
// profiling event pair around one launch and counts it.
void launch_begin(int kind, cudaStream_t s);
int launch_end(int kind, cudaStream_t s);  // returns SSD_OK or SSD_ERR_CUDA

// Stage launchers (one .cu file each).  Arguments are validated by the caller.
// A "span" is a run of `span_chunks` whole chunks; the stage entry points use
// one-chunk spans, ssd_forward uses longer ones.  `err` is the device error word.
int launch_chunk_cumsum(const float* dt, const float* A, const Dims& d, float* cs, float* dtt,
                        cudaStream_t s);
// chunk_cumsum plus, in the same launch, the float16 copies of B and C
// (the range flag of `err` is raised if a copied value exceeds float16's range)
int launch_chunk_cumsum_bc(const float* dt, const float* A, const Dims& d, float* cs, float* dtt,
                           const __nv_bfloat16* B, const __nv_bfloat16* C, __half* B16, __half* C16, int* err,
                           cudaStream_t s, const DtOpts& dto = DtOpts());
// B, C (bf16) -> float16 copies for the tensor-core products (see k_convert.cu)
int launch_bc_to_f16(const __nv_bfloat16* B, const __nv_bfloat16* C, const Dims& d, __half* B16, __half* C16,
                     int* err, cudaStream_t s);
// B and C below are the float16 copies; x stays bfloat16.
// S16: the span states written as float16 there instead of float32 to S (range flag in ctl.err)
// Heads of one B group that a chunk_state CTA covers (they share its B tile): 4, 2 or 1.
int chunk_state_heads_per_cta(const Dims& d);
int launch_chunk_state_span(const __nv_bfloat16* x, const __half* B, const float* dtt, const float* cs,
                            int span_chunks, const Dims& d, float* S, float* span_decay, const Ctl& ctl,
                            cudaStream_t s, __half* S16 = nullptr);
int launch_state_passing(const float* S, const float* cs, const float* init, const Dims& d,
                         float* states, float* final_state, cudaStream_t s);
// rev = 1: the steps run from the last to the first (the backward pass's hop, k_state_passing.cu);
// states16: the per-step states written as float16 there instead of float32 to `states` (range flag in err);
// S16: the per-step terms read as float16 from there instead of float32 from S
int launch_state_passing_steps(const float* S, const float* dec, int64_t dec_step, int64_t dec_row,
                               const float* init, const Dims& d, int nsteps, float* states, float* final_state,
                               cudaStream_t s, int rev = 0, __half* states16 = nullptr, int* err = nullptr,
                               const __half* S16 = nullptr);
// reverse-time chunk states for the backward pass (one-chunk spans): Z[c] = sum_t C_t 2^(cs(t)) dy_t^T
int launch_chunk_state_rev(const __nv_bfloat16* dy, const __half* C16, const float* dtt, const float* cs, const Dims& d,
                           float* Z, const Ctl& ctl, cudaStream_t s, __half* Z16 = nullptr);
// span_states holds one state per span of `span_chunks` chunks; chunk_scan walks spans of
// span_chunks * state_step chunks, each starting from every state_step-th of those states.
int launch_chunk_scan_span(const __nv_bfloat16* x, const __half* B, const __half* C,
                           const float* dtt, const float* cs, const float* D, const float* span_states,
                           int span_chunks, const Dims& d, __nv_bfloat16* y, const Ctl& ctl, cudaStream_t s,
                           const OutOpts& oo = OutOpts(), int state_step = 1);

// compute_out for two heads of one group per CTA (k_chunk_scan_pair.cu): state sizes 64 and 128, an
// even number of heads per group, no per-channel D or gate; launch_chunk_scan_span picks it when
// chunk_scan_pair_supported says so
bool chunk_scan_pair_supported(const Dims& d, const OutOpts& oo);
int launch_chunk_scan_pair(const __nv_bfloat16* x, const __half* B, const __half* C, const float* dtt,
                           const float* cs, const float* D, const float* span_states, int span_chunks, const Dims& d,
                           __nv_bfloat16* y, const Ctl& ctl, cudaStream_t s, int state_step);

// Backward pass (k_bwd.cu), over blocks of kBwdBlock tokens (d.chunk_size == kBwdBlock, d.nchunks blocks):
// per (block, group, batch) the gradients of every head of the group -- split over `slices` CTAs (a
// cluster; 1, 2 or 4, dividing the heads per group) -- from the block-start states h0
// and the block-end gradients mu (both (b, nblk, H, P, N) float16): dx, ddt, this block's rows of dB and
// dC (summed over the group's heads), and per (b, h, block) the partial sums of dt dl (for dA) and of
// x . dy (for dD), (b, H, nblk) f32 each.
constexpr int kBwdBlock = 128;
bool bwd_supported(const Dims& d);
int launch_bwd_chunk(const __nv_bfloat16* x, const __nv_bfloat16* dy, const __half* B16, const __half* C16,
                     const float* cs, const float* dtt, const float* A, const float* D, const __half* h0, const __half* mu,
                     const Dims& d, __nv_bfloat16* dx, float* ddt, float* dB, float* dC, float* dap, float* xdy,
                     const Ctl& ctl, cudaStream_t s, int slices);
// dA[h] and dD[h] (dD may be null): the partial sums over batch and blocks, in a fixed order
int launch_bwd_reduce(const float* dap, const float* xdy, const Dims& d, float* dA, float* dD, cudaStream_t s);

// one recurrent step for every (batch, head): state updated in place, y for the token (k_step.cu)
int launch_step(const __nv_bfloat16* x, const float* dt, const float* A, const __nv_bfloat16* B,
                const __nv_bfloat16* C, const float* D, float* state, int batch, int nheads, int ngroups, int dstate,
                __nv_bfloat16* y, cudaStream_t s, const DtOpts& dto = DtOpts(), const OutOpts& oo = OutOpts());
// ntok consecutive tokens of every sequence, the state in registers throughout (k_step.cu)
int launch_step_multi(const __nv_bfloat16* x, const float* dt, const float* A, const __nv_bfloat16* B,
                      const __nv_bfloat16* C, const float* D, float* state, int batch, int ntok, int nheads,
                      int ngroups, int dstate, __nv_bfloat16* y, cudaStream_t s);

}  // namespace ssd
