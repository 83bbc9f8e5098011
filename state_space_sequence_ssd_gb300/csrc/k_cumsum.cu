// k_cumsum.cu -- chunk_cumsum stage.
//
// devotd.net page on the Mamba-2 cuTile forward kernels, section 2 (the
// chunk_cumsum listing: a zero-padded (1, Q, BLOCK_H) tile of dt and a
// (BLOCK_H,) tile of A, cumulative sum of A*dt along the chunk, times log2 e)
// and section 3 (dA_cumsum and dt re-laid out for contiguous reads).
//
// One CTA per (chunk, 32-head tile, batch).  The (Q x 32) dt tile of a chunk
// is a run of Q rows of 32 contiguous floats, read coalesced into shared
// memory; each warp then scans 4 heads along the chunk (each lane owns Q/32
// consecutive positions: serial in-lane prefix + warp-shuffle scan of the
// lane totals) and writes the (batch, H, nchunks, Q) rows contiguously.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerCta = 32;
constexpr int kThreads = 256;

template <int Q>
__global__ void __launch_bounds__(kThreads) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                                const float* __restrict__ A, Dims d,
                                                                float* __restrict__ cs,
                                                                float* __restrict__ dtt) {
    __shared__ float tile[Q][kHeadsPerCta + 1];
    const int c = blockIdx.x, h0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // coalesced load: row i (token c*Q+i), column hh (head h0+hh)
    for (int i = tid >> 5; i < Q; i += kThreads / 32) {
        const int64_t t = (int64_t)c * Q + i;
        const int h = h0 + lane;
        float v = 0.f;
        if (t < d.seqlen && h < d.nheads) v = __ldg(dt + ((int64_t)b * d.seqlen + t) * d.nheads + h);
        tile[i][lane] = v;
    }
    __syncthreads();
    constexpr int kPer = Q / 32;  // positions per lane
    for (int hh = warp; hh < kHeadsPerCta; hh += kThreads / 32) {
        const int h = h0 + hh;
        if (h >= d.nheads) break;
        const float a = __ldg(A + h);
        float v[kPer], run = 0.f;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            v[k] = tile[lane * kPer + k][hh];
            run += a * v[k];
            v[k] = run;  // in-lane inclusive prefix of a*dt
        }
        // inclusive warp scan of the lane totals
        float tot = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, tot, off);
            if (lane >= off) tot += o;
        }
        const float excl = tot - run;
        const int64_t row = (((int64_t)b * d.nheads + h) * d.nchunks + c) * Q + lane * kPer;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            cs[row + k] = (v[k] + excl) * kLog2e;
            dtt[row + k] = tile[lane * kPer + k][hh];
        }
    }
}

}  // namespace

int launch_chunk_cumsum(const float* dt, const float* A, const Dims& d, float* cs, float* dtt,
                        cudaStream_t s) {
    dim3 grid(d.nchunks, ceil_div(d.nheads, kHeadsPerCta), d.batch);
    launch_begin(kKindCumsum, s);
    switch (d.chunk_size) {
        case 64: chunk_cumsum_kernel<64><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt); break;
        case 128: chunk_cumsum_kernel<128><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt); break;
        case 256: chunk_cumsum_kernel<256><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt); break;
        default: return SSD_ERR_UNSUPPORTED;
    }
    return launch_end(kKindCumsum, s);
}

}  // namespace ssd
