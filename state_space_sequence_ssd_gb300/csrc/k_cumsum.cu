// k_cumsum.cu -- chunk_cumsum stage.
//
// devotd.net page on the Mamba-2 cuTile forward kernels, section 2 (the
// chunk_cumsum listing: a zero-padded (1, Q, BLOCK_H) tile of dt and a
// (BLOCK_H,) tile of A, cumulative sum of A*dt along the chunk, times log2 e)
// and section 3 (dA_cumsum and dt re-laid out for contiguous reads).
//
// One CTA per (chunk, 8-head tile, batch).  The (Q x 8) dt tile is read with
// one pair of 16-byte loads per token row into shared memory; each warp then
// scans one head along the chunk (each lane owns Q/32 consecutive positions:
// serial in-lane prefix + warp-shuffle scan of the lane totals) and writes
// its (batch, H, nchunks, Q) rows through its tile row, each store instruction
// covering 512 contiguous bytes.
//
// With a layer's input-side options the dt tile is transformed as it is read
// (bias, softplus, clamp), so dt_t and every later stage see the effective dt.
//
// Optionally the same launch also writes the float16 copies of B and C that
// the tensor-core stages use (k_convert.cu explains why): the B/C elements
// are split evenly over all CTAs of the grid.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kHeads = 8;
constexpr int kThreads = 256;

// two bfloat16 -> two float16, saturating; mx tracks the largest magnitude seen (for the range flag)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t v, float& mx) {
    const float lo = __uint_as_float(v << 16);
    const float hi = __uint_as_float(v & 0xffff0000u);
    mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
    const __half2 h = __floats2half2_rn(fminf(fmaxf(lo, -kF16Max), kF16Max), fminf(fmaxf(hi, -kF16Max), kF16Max));
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 cvt16(const uint4& v, float& mx) {
    return make_uint4(bf16x2_to_f16x2_sat(v.x, mx), bf16x2_to_f16x2_sat(v.y, mx), bf16x2_to_f16x2_sat(v.z, mx),
                      bf16x2_to_f16x2_sat(v.w, mx));
}

// The B / C rows (batch, token) the copy covers, in 16-byte chunks: columns [col0, col0 + ncol) of rows
// of row16 chunks -- the groups of the call's heads (all of them for a whole-problem call: ncol == row16).
struct BcSpan {
    int64_t row16, col0, ncol;
    __device__ __forceinline__ int64_t offset(int64_t i) const {
        if (ncol == row16) return i;
        if (i < 0xffffffffll) {  // 32-bit division where it fits
            const uint32_t q = (uint32_t)i / (uint32_t)ncol;
            return (int64_t)q * row16 + col0 + ((uint32_t)i - q * (uint32_t)ncol);
        }
        return (i / ncol) * row16 + col0 + i % ncol;
    }
};

template <int Q>
__global__ void __launch_bounds__(kThreads) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                                const float* __restrict__ A, Dims d,
                                                                float* __restrict__ cs, float* __restrict__ dtt,
                                                                const uint4* __restrict__ bsrc,
                                                                const uint4* __restrict__ csrc, uint4* __restrict__ bdst,
                                                                uint4* __restrict__ cdst, int64_t bc16, BcSpan bsp,
                                                                int* err, DtOpts dto) {
    // tile[h][i + i / 8]: one padding word per 8 positions, so that lanes reading runs of
    // consecutive positions spread over the banks
    __shared__ float tile[kHeads][Q + Q / 8];
    // h0: first local head of this CTA (the call's intermediates); hg0 = h0 + head0 indexes dt, A, dt_bias
    const int c = blockIdx.x, h0 = blockIdx.y * kHeads, b = blockIdx.z;
    const int hg0 = d.head0 + h0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    grid_dep_launch_dependents();  // the next stage may set itself up while this one runs
    // this CTA's share of the B / C float16 copies (16-byte chunks); the first round of loads
    // is issued before the dt tile, so the two memory latencies overlap
    int64_t i = 0, hi = 0;
    uint4 vb[4], vc[4];
    bool first = false;
    if (bc16 > 0) {
        const int64_t nblk = (int64_t)gridDim.x * gridDim.y * gridDim.z;
        const int64_t blk = ((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        const int64_t per = (bc16 + nblk - 1) / nblk;
        const int64_t lo = blk * per;
        hi = min(bc16, lo + per);
        i = lo + tid;
        if (i + 3 * kThreads < hi) {
            first = true;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                vb[u] = __ldg(bsrc + bsp.offset(i + u * kThreads));
                vc[u] = __ldg(csrc + bsp.offset(i + u * kThreads));
            }
        }
    }
    // token row tid: 8 heads h0..h0+7
    if (tid < Q) {
        const int64_t t = (int64_t)c * Q + tid;
        float v[kHeads];
        if (t < d.seqlen) {
            const float* src = dt + ((int64_t)b * d.seqlen + t) * d.nheads + hg0;
            if (h0 + kHeads <= d.hcount && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
                const float4 a0 = __ldg(reinterpret_cast<const float4*>(src));
                const float4 a1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
                v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
                v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
            } else {
#pragma unroll
                for (int k = 0; k < kHeads; ++k) v[k] = (h0 + k < d.hcount) ? __ldg(src + k) : 0.f;
            }
            if (dto.active()) {  // the layer's dt transform, on real positions only (padding stays 0)
#pragma unroll
                for (int k = 0; k < kHeads; ++k)
                    if (h0 + k < d.hcount) v[k] = effective_dt(v[k], hg0 + k, dto);
            }
        } else {
#pragma unroll
            for (int k = 0; k < kHeads; ++k) v[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < kHeads; ++k) tile[k][tid + tid / 8] = v[k];
    }
    // the rest of the B / C share, independent of the scan
    if (bc16 > 0) {
        float mx = 0.f;
        for (; i + 3 * kThreads < hi; i += 4 * kThreads) {  // four chunks of B and C in flight
            if (!first) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    vb[u] = __ldg(bsrc + bsp.offset(i + u * kThreads));
                    vc[u] = __ldg(csrc + bsp.offset(i + u * kThreads));
                }
            }
            first = false;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t o = bsp.offset(i + u * kThreads);
                bdst[o] = cvt16(vb[u], mx);
                cdst[o] = cvt16(vc[u], mx);
            }
        }
        for (; i < hi; i += kThreads) {
            const int64_t o = bsp.offset(i);
            const uint4 vb = __ldg(bsrc + o), vc = __ldg(csrc + o);
            bdst[o] = cvt16(vb, mx);
            cdst[o] = cvt16(vc, mx);
        }
        flag_f16_range(err, mx);
    }
    __syncthreads();
    const int h = h0 + warp;
    if (h >= d.hcount) return;
    constexpr int kPer = Q / 32;  // positions per lane
    const float a = __ldg(A + d.head0 + h);
    float v[kPer], run = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pos = lane * kPer + k;
        const float x = tile[warp][pos + (pos >> 3)];
        run += a * x;
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
    // both rows leave through the warp's tile row, so that each store instruction writes 512 whole
    // bytes or the whole row (lane l: positions 4 l .. 4 l + 3 of every 128): first dt, then the cumsum
    const int64_t row = (((int64_t)b * d.hcount + h) * d.nchunks + c) * Q;
    float* trow = tile[warp];
    auto store_row = [&](float* dst) {
#pragma unroll
        for (int p = 4 * lane; p < Q; p += 128) {  // p .. p + 3 share one padded group of 8
            const float* t = trow + p + (p >> 3);
            *reinterpret_cast<float4*>(dst + row + p) = make_float4(t[0], t[1], t[2], t[3]);
        }
    };
    store_row(dtt);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pos = lane * kPer + k;
        trow[pos + (pos >> 3)] = (v[k] + excl) * kLog2e;
    }
    __syncwarp();
    store_row(cs);
}

}  // namespace

int launch_chunk_cumsum_bc(const float* dt, const float* A, const Dims& d, float* cs, float* dtt,
                           const __nv_bfloat16* B, const __nv_bfloat16* C, __half* B16, __half* C16, int* err,
                           cudaStream_t s, const DtOpts& dto) {
    dim3 grid(d.nchunks, ceil_div(d.hcount, kHeads), d.batch);
    // the groups of the call's heads
    const int hpg = d.nheads / d.ngroups;
    const int g0 = d.head0 / hpg, g1 = (d.head0 + d.hcount - 1) / hpg + 1;
    BcSpan bsp;
    bsp.row16 = (int64_t)d.ngroups * d.dstate / 8;
    bsp.col0 = (int64_t)g0 * d.dstate / 8;
    bsp.ncol = (int64_t)(g1 - g0) * d.dstate / 8;
    const int64_t bc16 = (B != nullptr) ? (int64_t)d.batch * d.seqlen * bsp.ncol : 0;
    const uint4* bs = reinterpret_cast<const uint4*>(B);
    const uint4* cs16 = reinterpret_cast<const uint4*>(C);
    uint4* bd = reinterpret_cast<uint4*>(B16);
    uint4* cd = reinterpret_cast<uint4*>(C16);
    launch_begin(kKindCumsum, s);
    switch (d.chunk_size) {
        case 64: chunk_cumsum_kernel<64><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt, bs, cs16, bd, cd, bc16, bsp, err, dto); break;
        case 128: chunk_cumsum_kernel<128><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt, bs, cs16, bd, cd, bc16, bsp, err, dto); break;
        case 256: chunk_cumsum_kernel<256><<<grid, kThreads, 0, s>>>(dt, A, d, cs, dtt, bs, cs16, bd, cd, bc16, bsp, err, dto); break;
        default: return SSD_ERR_UNSUPPORTED;
    }
    return launch_end(kKindCumsum, s);
}

int launch_chunk_cumsum(const float* dt, const float* A, const Dims& d, float* cs, float* dtt, cudaStream_t s) {
    return launch_chunk_cumsum_bc(dt, A, d, cs, dtt, nullptr, nullptr, nullptr, nullptr, nullptr, s);
}

}  // namespace ssd
