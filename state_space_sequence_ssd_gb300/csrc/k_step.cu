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
//
// The arithmetic runs two state entries per instruction (sm_100's packed two-lane float32 multiply
// and fma, each lane rounded as a separate instruction would be), and a lane's share of C.state is
// kept as two partial sums, of its even and of its odd entries, added at the end: the same order in
// every kernel here, so that K single steps and one K-token step agree bit for bit.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

// two float32 products, and two fused multiply-adds a * b + c, each in one instruction
__device__ __forceinline__ float2 pmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 pfma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// One state row's four entries of this lane: q <- a q + (dt B) x, then their terms of C.state added to
// the even / odd partial sums in acc
__device__ __forceinline__ void step4(float4& q, float a, float xp, const float (&bv)[4], const float (&cv)[4],
                                      float2& acc) {
    const float2 a2 = make_float2(a, a), x2 = make_float2(xp, xp);
    const float2 q01 = pfma2(a2, make_float2(q.x, q.y), pmul2(make_float2(bv[0], bv[1]), x2));
    const float2 q23 = pfma2(a2, make_float2(q.z, q.w), pmul2(make_float2(bv[2], bv[3]), x2));
    q = make_float4(q01.x, q01.y, q23.x, q23.y);
    acc = pfma2(make_float2(cv[0], cv[1]), q01, acc);
    acc = pfma2(make_float2(cv[2], cv[3]), q23, acc);
}

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
            float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float4 q = s4[i][v];
                step4(q, a, xp, bv[v], cv[v], acc2);
                *reinterpret_cast<float4*>(st + (int64_t)p * N + 128 * v + 4 * lane) = q;
            }
            float acc = acc2.x + acc2.y;
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
        float2 acc2 = make_float2(0.f, 0.f);
        step4(q, a, xp, bv, cv, acc2);
        *reinterpret_cast<float4*>(st + (int64_t)p * N + 4 * l16) = q;
        float acc = acc2.x + acc2.y;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (l16 == 0) y[bh * P + p] = __float2bfloat16_rn(step_output(acc, xp, Dh, h * P + p, bh * P + p, oo));
    }
}

// ---------------------------------------------------------------- several tokens per launch
// ssd_step_multi: K consecutive tokens of every sequence in one launch.  The state stays in
// registers for all K tokens, so it is read and written once per launch instead of once per
// token.  The tokens' inputs (dt, the B, C and x rows) come through shared memory in groups of KT
// tokens, copied asynchronously one group ahead, so one memory latency covers a group instead of
// each token paying its own.  Each token's arithmetic (the lanes' split of n, the packed state
// update, the two partial sums and the reduction order) is that of ssd_step, so K tokens here equal
// K ssd_step calls bit for bit.
// Sums R per-row partial values over the lanes of a row group (xor offsets OFF, OFF/2, ..., 1).
// While a lane holds more than one row it keeps half of them and trades the other half with its
// partner, so R rows over 2^k lanes cost (R - 1) + (k - log2 R) shuffles instead of R k (9 instead of
// 40 for 8 rows over 32 lanes).  Each
// row's sum is formed by the same butterfly pairings in the same order as a per-row xor reduction,
// so the result is bitwise the same.  On return the lane holds the full sum of row `row`.
template <int R, int OFF>
__device__ __forceinline__ float fold_rows(const float (&v)[R], int lane, int& row) {
    if constexpr (R == 1) {
        float t = v[0];
#pragma unroll
        for (int o = OFF; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        return t;
    } else {
        constexpr int HALF = R / 2;
        const bool up = (lane & OFF) != 0;
        float w[HALF];
#pragma unroll
        for (int j = 0; j < HALF; ++j) {
            const float mine = up ? v[j + HALF] : v[j];
            const float other = up ? v[j] : v[j + HALF];
            w[j] = mine + __shfl_xor_sync(0xffffffffu, other, OFF);
        }
        if (up) row += HALF;
        return fold_rows<HALF, OFF / 2>(w, lane, row);
    }
}

template <int N>
struct MultiCfg {
    static constexpr int THREADS = (N == 512) ? 512 : 256;
    static constexpr int W = THREADS / 32;
    static constexpr int LPR = (N == 64) ? 16 : 32;  // lanes per state row
    static constexpr int RPS = 32 / LPR;             // rows of a warp per slot
    static constexpr int NV = N / (4 * LPR);         // float4 per lane per row
    static constexpr int SLOTS = 64 / (W * RPS);     // rows held by each lane
    static constexpr int XW = SLOTS * RPS;           // a warp's rows (consecutive): 8, or 4 for N = 512
    // tokens per staged group: their B, C and x rows and dt go to shared memory together (two groups,
    // one filling while the other is used), so one memory latency covers KT tokens
    static constexpr int KT = (N <= 128) ? 16 : (N == 256 ? 8 : 4);
    static constexpr int OFF_C = KT * N * 2, OFF_X = 2 * KT * N * 2, OFF_DT = OFF_X + KT * 64 * 2;
    static constexpr int SZ = OFF_DT + KT * 4;  // bytes per group buffer (a multiple of 16)
    static_assert(SZ % 16 == 0, "group buffer alignment");
};

// 4-byte asynchronous copy global -> shared
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int NPEND>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(NPEND) : "memory");
}

template <int N>
__global__ void __launch_bounds__(MultiCfg<N>::THREADS) ssd_step_multi_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ dt, const float* __restrict__ A,
    const __nv_bfloat16* __restrict__ B, const __nv_bfloat16* __restrict__ C, const float* __restrict__ D,
    float* __restrict__ state, int ntok, int nheads, int ngroups, __nv_bfloat16* __restrict__ y) {
    using K = MultiCfg<N>;
    constexpr int P = 64;
    extern __shared__ __align__(16) uint8_t sbuf[];
    const int h = blockIdx.x, b = blockIdx.y;
    const int g = h / (nheads / ngroups);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = lane / K::LPR, ln = lane % K::LPR;
    const int64_t bh = (int64_t)b * nheads + h;
    float* st = state + bh * (int64_t)P * N;
    // this lane's rows: slot i is row (warp SLOTS + i) RPS + sub, so a warp's rows are consecutive
    auto row = [&](int i) { return (warp * K::SLOTS + i) * K::RPS + sub; };
    // the rows of tokens k0 .. k0 + cnt - 1 into group buffer `buf`: 16-byte asynchronous copies when
    // every row starts on 16 bytes, else element by element
    const bool al = ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C) |
                      reinterpret_cast<uintptr_t>(x)) & 15) == 0;
    auto stage = [&](int buf, int k0, int cnt) {
        uint8_t* sb = sbuf + buf * K::SZ;
        const uint32_t ss = (uint32_t)__cvta_generic_to_shared(sb);
        constexpr int RB = N / 8;                 // 16-byte pieces of a B or C row
        const int total = cnt * (2 * RB + 8);     // B, C and x pieces
        for (int c = tid; c < total; c += K::THREADS) {
            const int t = c / (2 * RB + 8), q = c % (2 * RB + 8);
            const int64_t bk = (int64_t)b * ntok + k0 + t;
            const __nv_bfloat16* src;
            uint32_t dst;
            if (q < RB) {
                src = B + (bk * ngroups + g) * N + q * 8;
                dst = t * N * 2 + q * 16;
            } else if (q < 2 * RB) {
                src = C + (bk * ngroups + g) * N + (q - RB) * 8;
                dst = K::OFF_C + t * N * 2 + (q - RB) * 16;
            } else {
                src = x + (bk * nheads + h) * P + (q - 2 * RB) * 8;
                dst = K::OFF_X + t * P * 2 + (q - 2 * RB) * 16;
            }
            if (al) {
                cp_async16(ss + dst, src);
            } else {
                __nv_bfloat16* d = reinterpret_cast<__nv_bfloat16*>(sb + dst);
#pragma unroll
                for (int e = 0; e < 8; ++e) d[e] = src[e];
            }
        }
        if (tid < cnt) cp_async4(ss + K::OFF_DT + 4 * tid, dt + ((int64_t)b * ntok + k0 + tid) * nheads + h);
        cp_async_commit();
    };
    stage(0, 0, ntok < K::KT ? ntok : K::KT);
    float4 s[K::SLOTS][K::NV];
#pragma unroll
    for (int i = 0; i < K::SLOTS; ++i)
#pragma unroll
        for (int v = 0; v < K::NV; ++v)
            s[i][v] = *reinterpret_cast<const float4*>(st + (int64_t)row(i) * N + 4 * ln + v * 4 * K::LPR);
    const float Ah = A[h];
    const float Dh = (D != nullptr) ? D[h] : 0.f;
#pragma unroll 1
    for (int k0 = 0, j = 0; k0 < ntok; k0 += K::KT, ++j) {
        const int cnt = (ntok - k0 < K::KT) ? ntok - k0 : K::KT;
        if (k0 + K::KT < ntok) {  // the next group fills the other buffer while this one is used
            stage((j + 1) & 1, k0 + K::KT, (ntok - k0 - K::KT < K::KT) ? ntok - k0 - K::KT : K::KT);
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        __syncthreads();  // every thread's copies of this group have landed
        const uint8_t* sb = sbuf + (j & 1) * K::SZ;
#pragma unroll 1
        for (int kk = 0; kk < cnt; ++kk) {
            const int64_t bk = (int64_t)b * ntok + k0 + kk;  // (batch, token) row of the (batch, K, ...) layouts
            const float dtv = reinterpret_cast<const float*>(sb + K::OFF_DT)[kk];
            const float a = expf(dtv * Ah);
            const __nv_bfloat16* Bg = reinterpret_cast<const __nv_bfloat16*>(sb + kk * N * 2);
            const __nv_bfloat16* Cg = reinterpret_cast<const __nv_bfloat16*>(sb + K::OFF_C + kk * N * 2);
            float bv[K::NV][4], cv[K::NV][4];
#pragma unroll
            for (int v = 0; v < K::NV; ++v) {
                const int n0 = 4 * ln + v * 4 * K::LPR;
                const uint2 bq = *reinterpret_cast<const uint2*>(Bg + n0);  // four bf16 in one 8-byte load
                const uint2 cq = *reinterpret_cast<const uint2*>(Cg + n0);
                const uint32_t bw[2] = {bq.x, bq.y}, cw[2] = {cq.x, cq.y};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    bv[v][e] = __uint_as_float((e & 1) ? (bw[e >> 1] & 0xffff0000u) : (bw[e >> 1] << 16)) * dtv;
                    cv[v][e] = __uint_as_float((e & 1) ? (cw[e >> 1] & 0xffff0000u) : (cw[e >> 1] << 16));
                }
            }
            // the warp's consecutive x values in one load (the same for all its lanes)
            const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(sb + K::OFF_X + kk * P * 2) +
                                      warp * K::XW;
            __nv_bfloat16 xw[K::XW];
            if constexpr (K::XW == 8) {
                *reinterpret_cast<uint4*>(xw) = *reinterpret_cast<const uint4*>(xs);
            } else {
                *reinterpret_cast<uint2*>(xw) = *reinterpret_cast<const uint2*>(xs);
            }
            __nv_bfloat16* yr = y + (bk * nheads + h) * P;
            float xp[K::SLOTS], acc[K::SLOTS];
#pragma unroll
            for (int i = 0; i < K::SLOTS; ++i) {
                xp[i] = __bfloat162float(xw[i * K::RPS + sub]);
                float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int v = 0; v < K::NV; ++v) step4(s[i][v], a, xp[i], bv[v], cv[v], acc2);
                acc[i] = acc2.x + acc2.y;
            }
            int i = 0;  // the row (slot) whose full sum this lane ends up holding
            const float tot = fold_rows<K::SLOTS, K::LPR / 2>(acc, ln, i);
            float xi = xp[0];
#pragma unroll
            for (int j2 = 1; j2 < K::SLOTS; ++j2) xi = (i == j2) ? xp[j2] : xi;
            if ((ln & (K::LPR / K::SLOTS - 1)) == 0)
                yr[row(i)] = __float2bfloat16_rn(step_output(tot, xi, Dh, 0, 0, OutOpts()));
        }
        __syncthreads();  // this buffer is refilled two groups on
    }
#pragma unroll
    for (int i = 0; i < K::SLOTS; ++i)
#pragma unroll
        for (int v = 0; v < K::NV; ++v)
            *reinterpret_cast<float4*>(st + (int64_t)row(i) * N + 4 * ln + v * 4 * K::LPR) = s[i][v];
}

}  // namespace

int launch_step_multi(const __nv_bfloat16* x, const float* dt, const float* A, const __nv_bfloat16* B,
                      const __nv_bfloat16* C, const float* D, float* state, int batch, int ntok, int nheads,
                      int ngroups, int dstate, __nv_bfloat16* y, cudaStream_t s) {
    // one token: the one-token kernel (the same arithmetic and bits; nothing to stage)
    if (ntok == 1) return launch_step(x, dt, A, B, C, D, state, batch, nheads, ngroups, dstate, y, s, DtOpts(), OutOpts());
    dim3 grid(nheads, batch);
    launch_begin(kKindStep, s);
    switch (dstate) {
        case 64:
            ssd_step_multi_kernel<64><<<grid, MultiCfg<64>::THREADS, 2 * MultiCfg<64>::SZ, s>>>(x, dt, A, B, C, D, state, ntok, nheads,
                                                                             ngroups, y);
            break;
        case 128:
            ssd_step_multi_kernel<128><<<grid, MultiCfg<128>::THREADS, 2 * MultiCfg<128>::SZ, s>>>(x, dt, A, B, C, D, state, ntok,
                                                                               nheads, ngroups, y);
            break;
        case 256:
            ssd_step_multi_kernel<256><<<grid, MultiCfg<256>::THREADS, 2 * MultiCfg<256>::SZ, s>>>(x, dt, A, B, C, D, state, ntok,
                                                                               nheads, ngroups, y);
            break;
        case 512:
            ssd_step_multi_kernel<512><<<grid, MultiCfg<512>::THREADS, 2 * MultiCfg<512>::SZ, s>>>(x, dt, A, B, C, D, state, ntok,
                                                                               nheads, ngroups, y);
            break;
        default: return SSD_ERR_UNSUPPORTED;
    }
    return launch_end(kKindStep, s);
}

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
