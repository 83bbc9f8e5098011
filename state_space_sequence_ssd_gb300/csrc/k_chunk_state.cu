// k_chunk_state.cu -- first half of fwd_pass_state: each chunk's own state.
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile", jump-formula paragraph: without
// decay the state advances by B X^T over a chunk (B, X the stacked per-token
// vectors); with decay, X's rows are pre-multiplied by exponentials of the
// log-space sums, which keeps the matrix-product form:
//
//   S[b,c,h][p][n] = sum_i B[t_i, g, n] * w_i * x[t_i, h, p],
//   w_i = 2^(cs[Q-1] - cs[i]) * dt_i            (cs, dt from chunk_cumsum)
//
// SIMT formulation: one CTA per (chunk, head, batch, 128-wide n tile); each
// thread accumulates an 8 (p) x 4 (n) fp32 tile over the chunk's tokens,
// staged 32 tokens at a time through shared memory.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTok = 32;     // tokens per shared-memory stage
constexpr int kNTile = 128;  // n columns per CTA
constexpr int kP = 64;       // headdim

__global__ void __launch_bounds__(kThreads) chunk_state_simt_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ B,
    const float* __restrict__ dtt, const float* __restrict__ cs, Dims d, float* __restrict__ S) {
    __shared__ float xs[kTok][kP + 4];
    __shared__ float bs[kTok][kNTile + 4];
    const int c = blockIdx.x, h = blockIdx.y % d.nheads, ntile = blockIdx.y / d.nheads, b = blockIdx.z;
    const int Q = d.chunk_size, N = d.dstate, H = d.nheads, G = d.ngroups;
    const int g = h / (H / G);
    const int n0 = ntile * kNTile;
    const int ncols = min(kNTile, N - n0);
    const int tid = threadIdx.x;
    const int pg = tid / 32, ng = tid % 32;  // p rows pg*8..+7, n cols ng*4..+3
    const float* csr = cs + (((int64_t)b * H + h) * d.nchunks + c) * Q;
    const float* dtr = dtt + (((int64_t)b * H + h) * d.nchunks + c) * Q;
    const float cs_last = csr[Q - 1];
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < Q; k0 += kTok) {
        __syncthreads();
        // x tile, scaled by w
        for (int e = tid; e < kTok * kP; e += kThreads) {
            const int k = e / kP, p = e % kP;
            const int64_t t = (int64_t)c * Q + k0 + k;
            float v = 0.f;
            if (t < d.seqlen) {
                const float w = exp2f(cs_last - csr[k0 + k]) * dtr[k0 + k];
                v = w * __bfloat162float(x[(((int64_t)b * d.seqlen + t) * H + h) * kP + p]);
            }
            xs[k][p] = v;
        }
        for (int e = tid; e < kTok * kNTile; e += kThreads) {
            const int k = e / kNTile, n = e % kNTile;
            const int64_t t = (int64_t)c * Q + k0 + k;
            float v = 0.f;
            if (t < d.seqlen && n < ncols) v = __bfloat162float(B[(((int64_t)b * d.seqlen + t) * G + g) * N + n0 + n]);
            bs[k][n] = v;
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < kTok; ++k) {
            float xv[8], bv[4];
#pragma unroll
            for (int i = 0; i < 8; ++i) xv[i] = xs[k][pg * 8 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = bs[k][ng * 4 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], bv[j], acc[i][j]);
        }
    }
    if (ng * 4 < ncols) {
        float* out = S + (((int64_t)b * d.nchunks + c) * H + h) * kP * N;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = pg * 8 + i;
            *reinterpret_cast<float4*>(out + (int64_t)p * N + n0 + ng * 4) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
}

}  // namespace

int launch_chunk_state(const __nv_bfloat16* x, const __nv_bfloat16* B, const float* dtt,
                       const float* cs, const Dims& d, float* S, cudaStream_t s) {
    dim3 grid(d.nchunks, d.nheads * ceil_div(d.dstate, kNTile), d.batch);
    launch_begin(kKindChunkState, s);
    chunk_state_simt_kernel<<<grid, kThreads, 0, s>>>(x, B, dtt, cs, d, S);
    return launch_end(kKindChunkState, s);
}

}  // namespace ssd
