// k_chunk_scan.cu -- compute_out: the chunk's output from its start state.
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile", three-kernel paragraph
// (carried-state term + decayed, causally masked interaction matrix + skip
// connection, fused in one tiled kernel); devotd.net page, section 2 (the
// intermediate matrix stays on chip instead of going to global memory).
//
//   y_i = 2^(cs_i) (C_i . h_c) + sum_{j<=i} (C_i . B_j) 2^(cs_i - cs_j) dt_j x_j + D x_i
//
// SIMT formulation: one CTA per (chunk, head, batch, 64-row tile).  The
// 64 x 64 interaction tiles are built in shared memory (never in global
// memory); each thread owns a 4 (row) x 4 (p) output tile.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;
constexpr int kP = 64;
constexpr int kNB = 32;  // n block for the state term

struct ScanSmem {
    // dynamic layout: Cs[kRows][N] bf16, Bs[kRows][N] bf16, Xs[64][68] f32,
    // Ms[64][68] f32, Ss[kNB][68] f32, csv[Q], dtv[Q]
    static size_t bytes(int N, int Q) {
        return (size_t)kRows * N * 2 * 2 + 64 * 68 * 4 * 2 + kNB * 68 * 4 + 2 * (size_t)Q * 4;
    }
};

__global__ void __launch_bounds__(kThreads) chunk_scan_simt_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ B,
    const __nv_bfloat16* __restrict__ C, const float* __restrict__ dtt, const float* __restrict__ cs,
    const float* __restrict__ D, const float* __restrict__ states, Dims d,
    __nv_bfloat16* __restrict__ y) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int Q = d.chunk_size, N = d.dstate, H = d.nheads, G = d.ngroups;
    const int rtiles = Q / kRows;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z / rtiles, rt = blockIdx.z % rtiles;
    const int g = h / (H / G);
    __nv_bfloat16* Cs = reinterpret_cast<__nv_bfloat16*>(smem);
    __nv_bfloat16* Bs = Cs + kRows * N;
    float* Xs = reinterpret_cast<float*>(Bs + kRows * N);
    float* Ms = Xs + 64 * 68;
    float* Ss = Ms + 64 * 68;
    float* csv = Ss + kNB * 68;
    float* dtv = csv + Q;
    const int tid = threadIdx.x;
    const int rg = tid / 16, pg = tid % 16;  // rows rg*4..+3, p (or j) pg*4..+3
    const int r0 = rt * kRows;                // first row of this tile inside the chunk
    const int64_t tchunk = (int64_t)c * Q;
    const int64_t rowbase = ((int64_t)b * H + h) * d.nchunks + c;

    for (int i = tid; i < Q; i += kThreads) {
        csv[i] = cs[rowbase * Q + i];
        dtv[i] = dtt[rowbase * Q + i];
    }
    // C rows of this tile
    for (int e = tid; e < kRows * N; e += kThreads) {
        const int i = e / N, n = e % N;
        const int64_t t = tchunk + r0 + i;
        Cs[e] = (t < d.seqlen) ? C[(((int64_t)b * d.seqlen + t) * G + g) * N + n] : __float2bfloat16(0.f);
    }
    __syncthreads();

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    // carried-state term: sum_n C[i,n] * state[p][n]
    const float* st = states + (((int64_t)b * d.nchunks + c) * H + h) * (int64_t)kP * N;
    for (int n0 = 0; n0 < N; n0 += kNB) {
        __syncthreads();
        for (int e = tid; e < kNB * kP; e += kThreads) {
            const int p = e / kNB, k = e % kNB;
            Ss[k * 68 + p] = st[(int64_t)p * N + n0 + k];
        }
        __syncthreads();
        for (int k = 0; k < kNB; ++k) {
            float cv[4], sv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cv[i] = __bfloat162float(Cs[(rg * 4 + i) * N + n0 + k]);
#pragma unroll
            for (int j = 0; j < 4; ++j) sv[j] = Ss[k * 68 + pg * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(cv[i], sv[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float e = exp2f(csv[r0 + rg * 4 + i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] *= e;
    }

    // intra-chunk term over column tiles j0 <= r0 (causal)
    for (int j0 = 0; j0 <= r0; j0 += kRows) {
        __syncthreads();
        for (int e = tid; e < kRows * N; e += kThreads) {
            const int j = e / N, n = e % N;
            const int64_t t = tchunk + j0 + j;
            Bs[e] = (t < d.seqlen) ? B[(((int64_t)b * d.seqlen + t) * G + g) * N + n] : __float2bfloat16(0.f);
        }
        for (int e = tid; e < 64 * kP; e += kThreads) {
            const int j = e / kP, p = e % kP;
            const int64_t t = tchunk + j0 + j;
            Xs[j * 68 + p] = (t < d.seqlen) ? __bfloat162float(x[(((int64_t)b * d.seqlen + t) * H + h) * kP + p]) : 0.f;
        }
        __syncthreads();
        // CB tile: rows rg*4.., cols pg*4..
        float cb[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) cb[i][j] = 0.f;
        for (int n = 0; n < N; ++n) {
            float cv[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cv[i] = __bfloat162float(Cs[(rg * 4 + i) * N + n]);
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = __bfloat162float(Bs[(pg * 4 + j) * N + n]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) cb[i][j] = fmaf(cv[i], bv[j], cb[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ri = r0 + rg * 4 + i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cj = j0 + pg * 4 + j;
                const bool valid = (cj <= ri) && (tchunk + cj < d.seqlen);
                Ms[(rg * 4 + i) * 68 + pg * 4 + j] = valid ? cb[i][j] * exp2f(csv[ri] - csv[cj]) * dtv[cj] : 0.f;
            }
        }
        __syncthreads();
        for (int j = 0; j < 64; ++j) {
            float mv[4], xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mv[i] = Ms[(rg * 4 + i) * 68 + j];
#pragma unroll
            for (int q = 0; q < 4; ++q) xv[q] = Xs[j * 68 + pg * 4 + q];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(mv[i], xv[q], acc[i][q]);
        }
    }

    const float Dh = (D != nullptr) ? D[h] : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = tchunk + r0 + rg * 4 + i;
        if (t >= d.seqlen) continue;
        const int64_t o = (((int64_t)b * d.seqlen + t) * H + h) * kP + pg * 4;
        __nv_bfloat16 out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) out[q] = __float2bfloat16_rn(acc[i][q] + Dh * __bfloat162float(x[o + q]));
        *reinterpret_cast<uint2*>(y + o) = *reinterpret_cast<uint2*>(out);
    }
}

}  // namespace

int launch_chunk_scan(const __nv_bfloat16* x, const __nv_bfloat16* B, const __nv_bfloat16* C,
                      const float* dtt, const float* cs, const float* D, const float* states,
                      const Dims& d, __nv_bfloat16* y, cudaStream_t s) {
    const size_t smem = ScanSmem::bytes(d.dstate, d.chunk_size);
    cudaError_t e = cudaFuncSetAttribute(chunk_scan_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    dim3 grid(d.nchunks, d.nheads, d.batch * (d.chunk_size / kRows));
    launch_begin(kKindChunkScan, s);
    chunk_scan_simt_kernel<<<grid, kThreads, smem, s>>>(x, B, C, dtt, cs, D, states, d, y);
    return launch_end(kKindChunkScan, s);
}

}  // namespace ssd
