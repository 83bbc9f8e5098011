// k_step.cu -- one recurrent step of the selective state-space model: the
// constant-memory per-token update that the chunked forward pass computes in
// bulk.
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile", SSM/attention/RNN paragraph (the
// model can run as a recurrence with a fixed-size state) and readmex.ai page,
// English excerpt (the sequence-model trade-off: constant memory per token).
// Per batch row b and head h (group g = h / (H / G)), for the single token:
//
//   a              = exp(dt A_h)
//   state[p][n]   <- a state[p][n] + dt B[n] x[p]
//   y[p]           = sum_n C[n] state[p][n] + D_h x[p]
//
// One CTA per (b, h), 256 threads: warp w updates state rows p = w, w + 8, ...
// (each lane four consecutive n per 128 n, one float4 load and store per 128 n)
// and reduces the row's dot product with C by warp shuffles.  A warp issues the
// loads of its rows' state (up to 32 floats per lane) before anything else, so
// one memory latency covers them.  The state is read and written once: the
// step is bound by HBM.  fp32 throughout.
//
// With a layer's input-side options, dt is transformed first (bias, softplus,
// clamp), the skip weight may be one per channel (D is (H, P)) and y is gated
// by z sigmoid(z); the state itself is never gated.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// y = C.state + D x, then the optional gate; hp indexes (H, P) weights, i the (batch, H, P) rows
__device__ __forceinline__ float step_output(float acc, float xp, float Dh, int64_t hp, int64_t i, const OutOpts& oo) {
    float v = acc + ((oo.Dp != nullptr) ? oo.Dp[hp] : Dh) * xp;
    if (oo.z != nullptr) v *= silu(__bfloat162float(oo.z[i]));
    return v;
}

template <int N>
__global__ void __launch_bounds__(kThreads) ssd_step_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ dt,
                                                            const float* __restrict__ A,
                                                            const __nv_bfloat16* __restrict__ B,
                                                            const __nv_bfloat16* __restrict__ C,
                                                            const float* __restrict__ D, float* __restrict__ state,
                                                            int nheads, int ngroups, __nv_bfloat16* __restrict__ y,
                                                            DtOpts dto, OutOpts oo) {
    constexpr int P = 64;
    constexpr int NV = N / 128;        // float4 per lane per row
    constexpr int RG = 8 / NV;         // rows whose state is in flight at once (32 floats per lane)
    constexpr int ROWS = P / (kThreads / 32);  // rows per warp: p = warp + 8 i
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / (nheads / ngroups);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = (int64_t)b * nheads + h;
    float* st = state + bh * (int64_t)P * N;
    // the state loads go out first: they depend on nothing else
    float4 s4[RG][NV];
#pragma unroll
    for (int i = 0; i < RG; ++i)
#pragma unroll
        for (int v = 0; v < NV; ++v)
            s4[i][v] = *reinterpret_cast<const float4*>(st + (int64_t)(warp + 8 * i) * N + 128 * v + 4 * lane);
    const float dtv = dto.active() ? effective_dt(dt[bh], h, dto) : dt[bh];
    const float a = expf(dtv * A[h]);
    const float Dh = (D != nullptr) ? D[h] : 0.f;
    // this lane's B and C entries: n = 128 v + 4 lane + e (four bf16 in one 8-byte load)
    float bv[NV][4], cv[NV][4];
    const __nv_bfloat16* Bg = B + ((int64_t)b * ngroups + g) * N;
    const __nv_bfloat16* Cg = C + ((int64_t)b * ngroups + g) * N;
    const bool vec = ((reinterpret_cast<uintptr_t>(Bg) | reinterpret_cast<uintptr_t>(Cg)) & 7) == 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int n0 = 128 * v + 4 * lane;
        if (vec) {
            const uint2 bq = *reinterpret_cast<const uint2*>(Bg + n0);
            const uint2 cq = *reinterpret_cast<const uint2*>(Cg + n0);
            const uint32_t bw[2] = {bq.x, bq.y}, cw[2] = {cq.x, cq.y};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                bv[v][e] = __uint_as_float((e & 1) ? (bw[e >> 1] & 0xffff0000u) : (bw[e >> 1] << 16)) * dtv;
                cv[v][e] = __uint_as_float((e & 1) ? (cw[e >> 1] & 0xffff0000u) : (cw[e >> 1] << 16));
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                bv[v][e] = __bfloat162float(Bg[n0 + e]) * dtv;
                cv[v][e] = __bfloat162float(Cg[n0 + e]);
            }
        }
    }
    const __nv_bfloat16* xr = x + bh * P;
#pragma unroll
    for (int r0 = 0; r0 < ROWS; r0 += RG) {
        if (r0 > 0) {  // next group of rows (N >= 256)
#pragma unroll
            for (int i = 0; i < RG; ++i)
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    s4[i][v] = *reinterpret_cast<const float4*>(st + (int64_t)(warp + 8 * (r0 + i)) * N + 128 * v +
                                                                4 * lane);
        }
#pragma unroll
        for (int i = 0; i < RG; ++i) {
            const int p = warp + 8 * (r0 + i);
            const float xp = __bfloat162float(xr[p]);
            float acc = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float4 q = s4[i][v];
                q.x = fmaf(a, q.x, bv[v][0] * xp);
                q.y = fmaf(a, q.y, bv[v][1] * xp);
                q.z = fmaf(a, q.z, bv[v][2] * xp);
                q.w = fmaf(a, q.w, bv[v][3] * xp);
                *reinterpret_cast<float4*>(st + (int64_t)p * N + 128 * v + 4 * lane) = q;
                acc = fmaf(cv[v][0], q.x, acc);
                acc = fmaf(cv[v][1], q.y, acc);
                acc = fmaf(cv[v][2], q.z, acc);
                acc = fmaf(cv[v][3], q.w, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) y[bh * P + p] = __float2bfloat16_rn(step_output(acc, xp, Dh, h * P + p, bh * P + p, oo));
        }
    }
}

// N = 64: half a warp's lanes per row (each lane four n); a warp's eight rows are loaded up front.
__global__ void __launch_bounds__(kThreads) ssd_step_kernel_n64(const __nv_bfloat16* __restrict__ x,
                                                                const float* __restrict__ dt,
                                                                const float* __restrict__ A,
                                                                const __nv_bfloat16* __restrict__ B,
                                                                const __nv_bfloat16* __restrict__ C,
                                                                const float* __restrict__ D, float* __restrict__ state,
                                                                int nheads, int ngroups, __nv_bfloat16* __restrict__ y,
                                                                DtOpts dto, OutOpts oo) {
    constexpr int P = 64, N = 64;
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / (nheads / ngroups);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int64_t bh = (int64_t)b * nheads + h;
    float* st = state + bh * (int64_t)P * N;
    // the state loads go out first: they depend on nothing else
    constexpr int PAIRS = P / (2 * (kThreads / 32));  // row pairs per warp: p = 2 warp + 16 i + half
    float4 s4[PAIRS];
#pragma unroll
    for (int i = 0; i < PAIRS; ++i)
        s4[i] = *reinterpret_cast<const float4*>(st + (int64_t)(2 * warp + 16 * i + half) * N + 4 * l16);
    const float dtv = dto.active() ? effective_dt(dt[bh], h, dto) : dt[bh];
    const float a = expf(dtv * A[h]);
    const float Dh = (D != nullptr) ? D[h] : 0.f;
    const __nv_bfloat16* Bg = B + ((int64_t)b * ngroups + g) * N;
    const __nv_bfloat16* Cg = C + ((int64_t)b * ngroups + g) * N;
    float bv[4], cv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        bv[e] = __bfloat162float(Bg[4 * l16 + e]) * dtv;
        cv[e] = __bfloat162float(Cg[4 * l16 + e]);
    }
    const __nv_bfloat16* xr = x + bh * P;
#pragma unroll
    for (int i = 0; i < PAIRS; ++i) {
        const int p = 2 * warp + 16 * i + half;
        const float xp = __bfloat162float(xr[p]);
        float4 q = s4[i];
        q.x = fmaf(a, q.x, bv[0] * xp);
        q.y = fmaf(a, q.y, bv[1] * xp);
        q.z = fmaf(a, q.z, bv[2] * xp);
        q.w = fmaf(a, q.w, bv[3] * xp);
        *reinterpret_cast<float4*>(st + (int64_t)p * N + 4 * l16) = q;
        float acc = cv[0] * q.x;
        acc = fmaf(cv[1], q.y, acc);
        acc = fmaf(cv[2], q.z, acc);
        acc = fmaf(cv[3], q.w, acc);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (l16 == 0) y[bh * P + p] = __float2bfloat16_rn(step_output(acc, xp, Dh, h * P + p, bh * P + p, oo));
    }
}

}  // namespace

int launch_step(const __nv_bfloat16* x, const float* dt, const float* A, const __nv_bfloat16* B,
                const __nv_bfloat16* C, const float* D, float* state, int batch, int nheads, int ngroups, int dstate,
                __nv_bfloat16* y, cudaStream_t s, const DtOpts& dto, const OutOpts& oo) {
    dim3 grid(nheads, batch);
    launch_begin(kKindStep, s);
    switch (dstate) {
        case 64: ssd_step_kernel_n64<<<grid, kThreads, 0, s>>>(x, dt, A, B, C, D, state, nheads, ngroups, y, dto, oo); break;
        case 128: ssd_step_kernel<128><<<grid, kThreads, 0, s>>>(x, dt, A, B, C, D, state, nheads, ngroups, y, dto, oo); break;
        case 256: ssd_step_kernel<256><<<grid, kThreads, 0, s>>>(x, dt, A, B, C, D, state, nheads, ngroups, y, dto, oo); break;
        case 512: ssd_step_kernel<512><<<grid, kThreads, 0, s>>>(x, dt, A, B, C, D, state, nheads, ngroups, y, dto, oo); break;
        default: return SSD_ERR_UNSUPPORTED;
    }
    return launch_end(kKindStep, s);
}

}  // namespace ssd
