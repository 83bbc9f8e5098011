// k_chunk_state.cu -- first half of fwd_pass_state on tcgen05 tensor cores.
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile", jump-formula paragraph: with no
// decay a run of tokens advances the state by B^T X (B, X the stacked
// per-token vectors); with decay, X's rows are pre-scaled by exponentials of
// the log-space sums, which keeps one matrix product:
//
//   S_span[p][n] = sum_{t in span} B[t, n] * w_t * x[t, p],
//   w_t = 2^(cs_span_end - cs_span(t)) * dt_t
//
// A span is a run of whole chunks (one chunk for ssd_chunk_state).  With
// per-chunk cumsums cs[c][i] (chunk_cumsum's output), the exponent is
//   R_c + cs[c][Q-1] - cs[c][i],   R_c = sum of cs[c'][Q-1] over the span's chunks after c,
// every term <= 0, so no intermediate overflows.  The span's total exponent
// sum_c cs[c][Q-1] is also written (log2 decay of the whole span).
//
// One CTA per (HH heads of one B group, span, batch): the heads share the B
// tile and one MMA per k-step, whose N = 64 HH columns hold the HH heads'
// states side by side:
//   acc[mb] (128 n x 64 HH, f32 in TMEM) += B_tile^T (MN-major) * [X'_0 .. X'_HH-1] (MN-major).
// HH = 4 for N <= 128 and 2 for N >= 256 when the heads per group allow it
// (fewer and wider MMAs, one B load per HH heads).  Roles: one or two
// warpgroups scale the X rows in shared memory (one token row per thread)
// and store the result; one warp issues the TMA loads; one warp owns TMEM
// and issues the MMAs.
// Reverse-time mode (the backward pass, one-chunk spans): the same product with C in B's place,
// dy in x's place and w_t = 2^(cs(t)) (the decay from the chunk start through token t, no dt
// factor), which gives the chunk's contribution to the gradient flowing into the state before it:
//   Z_c[p][n] = sum_{t in chunk} C[t, n] * 2^(cs(t)) * dy[t, p].
// Operands are float16: B is the exact float16 copy of the input, and the
// scaled rows w x (bfloat16 x times an f32 weight) are rounded once to
// float16, whose 11 significant bits keep the state within tolerance.
#include "common.cuh"
#include "sm100.cuh"
#include "tmap.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kMaxSpanChunks = 256;

// HH heads of one B group per CTA: they share the B tile, and one MMA per
// k-step covers all of them (N = 64 HH).  2 scaling warpgroups when HH > 1.
// ONE: a grid of at most one CTA per SM, which then takes twice the shared memory for stages.
template <int N, int HH, bool ONE>
struct StCfg {
    static constexpr int TB = 64;                      // tokens per stage
    static constexpr int BOX = TB * 128;               // one 64-column box, TB rows
    static constexpr int NBOX = N / 64;                // boxes of B per stage
    static constexpr int MB = (N + 127) / 128;         // 128-row accumulator blocks
    static constexpr int SW = (HH > 1) ? 2 : 1;        // scaling warpgroups
    static constexpr int THREADS = 128 * SW + 64;      // + TMA warp + MMA warp
    static constexpr int WARP_TMA = 4 * SW, WARP_MMA = 4 * SW + 1;
    // per stage: HH x tiles, the B boxes, then HH x {cs[TB], dt[TB]}; 1024-byte aligned stages
    static constexpr int OFF_B = HH * BOX;
    static constexpr int OFF_CD = OFF_B + NBOX * BOX;
    static constexpr int SZ_STAGE = (OFF_CD + HH * 2 * TB * 4 + 1023) / 1024 * 1024;
    // as many stages as fit about 100 KB (two CTAs per SM) or 208 KB (one), 2 to 4: a stage refills
    // only after its MMAs retire, so more stages keep more of the x stream in flight
    static constexpr int NST_FIT = ((ONE ? 208 : 100) * 1024) / SZ_STAGE;
    static constexpr int NST = NST_FIT < 2 ? 2 : (NST_FIT > 4 ? 4 : NST_FIT);
    static constexpr int OFF_ZERO = NST * SZ_STAGE;
    static constexpr int SZ_ZERO = (N == 64) ? BOX : 0;  // zero rows padding the A operand to 128
    static constexpr int OFF_R = OFF_ZERO + SZ_ZERO;     // HH x per chunk of the span: R_c + cs[c][Q-1]
    static constexpr int OFF_BAR = OFF_R + HH * kMaxSpanChunks * 4;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    static constexpr int CTAS_PER_SM = (!ONE && SMEM <= 113 * 1024) ? 2 : 1;
    static constexpr int TCOLS = MB * HH * 64 <= 32 ? 32 : (MB * HH * 64 <= 64 ? 64 : (MB * HH * 64 <= 128 ? 128 : (MB * HH * 64 <= 256 ? 256 : 512)));
    static_assert(MB * HH * 64 <= 512, "TMEM budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct StateArgs {
    Dims d;
    int span_chunks;
    int nspans;
    const float* cs;    // (b, hcount, nc, Q)
    const float* dtt;   // (b, hcount, nc, Q)
    float* S;           // (b, nspans, hcount, P, N)
    __half* S16;        // the same as float16 instead, or null
    float* span_decay;  // (b, hcount, nspans) log2 units, or null
    Ctl ctl;            // error words, wait limit, stall hook
    int rev;            // reverse-time weights (one-chunk spans): w_t = 2^(cs(t)), no dt factor
};

template <int N, int HH, bool ONE>
__global__ void __launch_bounds__(StCfg<N, HH, ONE>::THREADS, StCfg<N, HH, ONE>::CTAS_PER_SM)
    chunk_state_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                          StateArgs a) {
    using K = StCfg<N, HH, ONE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
    uint64_t* xs_ready = full + K::NST;
    uint64_t* empty = xs_ready + K::NST;
    uint64_t* acc_done = empty + K::NST;
    uint64_t* stall_bar = acc_done + 1;  // never completed: the test hook's wait runs out on it
    float* Rs = reinterpret_cast<float*>(smem + K::OFF_R);  // head hh at hh * kMaxSpanChunks
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const Dims& d = a.d;
    // h0: first local head of the CTA (intermediates); hg0 = head0 + h0: its head in x and B
    const int h0 = blockIdx.x * HH, s = blockIdx.y, b = blockIdx.z;
    const int H = d.nheads, HC = d.hcount, G = d.ngroups, Q = d.chunk_size;
    const int hg0 = d.head0 + h0;
    const int g = hg0 / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ts = (int64_t)s * a.span_chunks * Q;
    const int64_t te = min((int64_t)d.seqlen, ts + (int64_t)a.span_chunks * Q);
    const int nblk = (int)((te - ts + K::TB - 1) / K::TB);
    const int64_t c_first = ts / Q;
    const int nchk = (int)((te - ts + Q - 1) / Q);
    const int64_t rowlen = (int64_t)d.nchunks * Q;  // dA_cumsum / dt row length per (b, h)

    if (threadIdx.x == 0) {
        for (int i = 0; i < K::NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&xs_ready[i], 128 * K::SW);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_done, 1);
        mbar_init(stall_bar, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    grid_dep_wait();  // dA_cumsum, dt and the float16 B come from the previous launch
    grid_dep_launch_dependents();
    if (K::SZ_ZERO > 0) {
        uint4* z = reinterpret_cast<uint4*>(smem + K::OFF_ZERO);
        for (int i = threadIdx.x; i < K::SZ_ZERO / 16; i += K::THREADS) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == K::WARP_MMA) {
        tmem_alloc(&tmem_base_sh, K::TCOLS);
        tmem_relinquish();
    }
    if (warp == K::WARP_TMA && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_B);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base_sh;
    volatile int* abort_flag = &abort_sh;
    int* const err = a.ctl.err;
    const uint64_t wait_ns = a.ctl.wait_ns;

    if (warp == K::WARP_TMA) {
        // TMA producer: per stage the HH x tiles, the B boxes and the heads' dA_cumsum / dt rows
        if (lane == 0) {
            if (a.ctl.stall) mbar_wait_bounded(stall_bar, 0, abort_flag, err, 20, wait_ns);
            int nissued = 0;  // stage loads issued; stage i took those with index % NST == i
            for (int kb = 0; kb < nblk && !*abort_flag; ++kb) {
                const int st = kb % K::NST;
                if (!mbar_wait_bounded_inline(&empty[st], ((kb / K::NST) & 1) ^ 1, abort_flag, err, 21, wait_ns)) break;
                uint8_t* sX = smem + st * K::SZ_STAGE;
                const int t0 = (int)(ts + (int64_t)kb * K::TB);
                const uint32_t cdb = (uint32_t)min((int64_t)K::TB, rowlen - t0) * 4u;
                float* scd = reinterpret_cast<float*>(sX + K::OFF_CD);
                mbar_arrive_expect_tx(&full[st], HH * K::BOX + K::NBOX * K::BOX + HH * 2 * cdb);
#pragma unroll
                for (int hh = 0; hh < HH; ++hh) {
                    const int64_t row = ((int64_t)b * HC + h0 + hh) * rowlen + t0;
                    tma_load_4d(sX + hh * K::BOX, &tm_x, &full[st], 0, hg0 + hh, t0, b);
                    bulk_load(scd + hh * 2 * K::TB, a.cs + row, cdb, &full[st]);
                    bulk_load(scd + hh * 2 * K::TB + K::TB, a.dtt + row, cdb, &full[st]);
                }
#pragma unroll
                for (int bx = 0; bx < K::NBOX; ++bx)
                    tma_load_4d(sX + K::OFF_B + bx * K::BOX, &tm_B, &full[st], bx * 64, g, t0, b);
                ++nissued;
            }
#pragma unroll
            for (int i = 0; i < K::NST; ++i) {  // every issued load has landed before teardown
                const int issued = (nissued + K::NST - 1 - i) / K::NST;
                if (issued > 0) mbar_wait_drain(&full[i], (issued - 1) & 1, err, 122, kDrainNs);
            }
        }
    } else if (warp == K::WARP_MMA) {
        // MMA issuer: acc[mb] (128 n x 64 HH) += B_mb^T (MN-major) * [X'_0 .. X'_HH-1] (MN-major)
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_fp16(128, 64 * HH, true, true);
            for (int kb = 0; kb < nblk; ++kb) {
                const int st = kb % K::NST;
                if (!mbar_wait_bounded_inline(&xs_ready[st], (kb / K::NST) & 1, abort_flag, err, 23, wait_ns)) break;
                tc_fence_after();
                const uint32_t sX = smem_u32(smem + st * K::SZ_STAGE);
                const uint32_t sB = sX + K::OFF_B;
#pragma unroll
                for (int mb = 0; mb < K::MB; ++mb) {
                    const uint32_t a0 = sB + 2 * mb * K::BOX;
                    const uint32_t lbo = (N == 64) ? (uint32_t)(smem_u32(smem + K::OFF_ZERO) - a0) : (uint32_t)K::BOX;
#pragma unroll
                    for (int k = 0; k < K::TB / 16; ++k)
                        mma_ss(tm + mb * 64 * HH, desc_sw128(a0 + k * 2048, lbo, 1024),
                               desc_sw128(sX + k * 2048, HH > 1 ? (uint32_t)K::BOX : 16u, 1024), idesc, (kb | k) != 0);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(acc_done);
            mbar_wait_drain(acc_done, 0, err, 125, kDrainNs);  // every product retired before TMEM is freed
        }
    } else {
        // scaling warpgroup(s): thread t scales token row t % TB of the x tiles of heads
        // hh = t / TB, t / TB + 128 SW / TB, ... in place; afterwards thread t stores TMEM lane t % 128.
        // First (not in reverse-time mode, which weights by 2^(cs) alone): warp hh < HH forms head
        // h0 + hh's R_c + cs[c][Q-1] per chunk c of the span -- the sum of the chunk totals from c to the
        // span end (an inclusive suffix sum), 32 chunks per round, one load per lane -- while the first
        // stages load.
        if (warp < HH && (!a.rev || a.span_decay != nullptr)) {
            const int64_t row = (int64_t)b * HC + h0 + warp;
            const float* csr = a.cs + row * rowlen;
            float carry = 0.f;
            for (int base = nchk - 32; base > -32; base -= 32) {
                const int c = base + lane;
                float v = (c >= 0) ? csr[(c_first + c) * Q + Q - 1] : 0.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {  // suffix scan: add the lanes above
                    const float o = __shfl_down_sync(0xffffffffu, v, off);
                    if (lane + off < 32) v += o;
                }
                v += carry;
                if (c >= 0) Rs[warp * kMaxSpanChunks + c] = v;
                carry = __shfl_sync(0xffffffffu, v, 0);
            }
            if (lane == 0 && a.span_decay != nullptr) a.span_decay[row * a.nspans + s] = carry;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(128 * K::SW) : "memory");  // the scaling warps only
        const int r = threadIdx.x & 127;
        const int hsel = threadIdx.x >> 7;
        const int rr = threadIdx.x % K::TB;
        constexpr int kHeadStep = 128 * K::SW / K::TB;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        float mx = 0.f;  // largest |w x| converted to float16 (range flag)
        for (int kb = 0; kb < nblk; ++kb) {
            const int st = kb % K::NST;
            ok = ok && mbar_wait_bounded_inline(&full[st], (kb / K::NST) & 1, abort_flag, err, 24, wait_ns);
            if (ok) {
                const int64_t t = ts + (int64_t)kb * K::TB + rr;
                uint8_t* stage = smem + st * K::SZ_STAGE;
                const float* scd = reinterpret_cast<const float*>(stage + K::OFF_CD);
#pragma unroll 1
                for (int hh = (int)(threadIdx.x / K::TB); hh < HH; hh += kHeadStep) {
                    uint8_t* xrow = stage + hh * K::BOX;
                    const float* cd = scd + hh * 2 * K::TB;
                    float w = 0.f;
                    if (t < te)
                        w = a.rev ? exp2f(cd[rr])
                                  : exp2f(Rs[hh * kMaxSpanChunks + (int)(t / Q - c_first)] - cd[rr]) * cd[K::TB + rr];
                    uint4 v[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) v[ch] = *reinterpret_cast<const uint4*>(xrow + sw128_offset(rr, ch));
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[ch]);
                        uint4 o;
                        __half2* o2 = reinterpret_cast<__half2*>(&o);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(p2[e]);
                            const float a0 = f.x * w, a1 = f.y * w;
                            mx = fmaxf(mx, fmaxf(fabsf(a0), fabsf(a1)));
                            o2[e] = __floats2half2_rn(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(xrow + sw128_offset(rr, ch)) = o;
                    }
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&xs_ready[st]);
        }
        flag_f16_range(err, mx);
        ok = ok && mbar_wait_bounded_inline(acc_done, 0, abort_flag, err, 25, wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (ok) {
            const int64_t PN = (int64_t)d.headdim * N;
            float smx = 0.f;  // largest |state| written as float16
#pragma unroll 1
            for (int hh = hsel; hh < HH; hh += K::SW) {
                const int64_t o = (((int64_t)b * a.nspans + s) * HC + h0 + hh) * PN;
#pragma unroll 1
                for (int mb = 0; mb < K::MB; ++mb) {
                    const int n = mb * 128 + r;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t v[32];
                        tmem_ld32(tm + lane_base + mb * 64 * HH + hh * 64 + half * 32, v);
                        tmem_ld_wait(v);
                        if (n < N) {
                            if (a.S16 != nullptr) {
                                __half* out = a.S16 + o;
#pragma unroll
                                for (int p = 0; p < 32; ++p) {
                                    const float f = __uint_as_float(v[p]);
                                    smx = fmaxf(smx, fabsf(f));
                                    out[(int64_t)(half * 32 + p) * N + n] = __float2half_rn(f);
                                }
                            } else {
                                float* out = a.S + o;
#pragma unroll
                                for (int p = 0; p < 32; ++p) out[(int64_t)(half * 32 + p) * N + n] = __uint_as_float(v[p]);
                            }
                        }
                    }
                }
            }
            flag_f16_range(err, smx);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == K::WARP_MMA) tmem_dealloc(tm, K::TCOLS);
}

template <int N, int HH, bool ONE>
int launch_state_nho(const __nv_bfloat16* x, const __half* B, const StateArgs& a, cudaStream_t s) {
    using K = StCfg<N, HH, ONE>;
    const Dims& d = a.d;
    CUtensorMap tx, tb;
    const uint64_t dx[4] = {(uint64_t)d.headdim, (uint64_t)d.nheads, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint64_t db[4] = {(uint64_t)d.dstate, (uint64_t)d.ngroups, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint32_t box[4] = {64, 1, (uint32_t)K::TB, 1};
    if (!make_tmap_16b_4d(&tx, x, dx, box) || !make_tmap_16b_4d(&tb, B, db, box)) return SSD_ERR_CUDA;
    if (ensure_smem_limit(reinterpret_cast<const void*>(chunk_state_tc_kernel<N, HH, ONE>), K::SMEM) != SSD_OK)
        return SSD_ERR_CUDA;
    dim3 grid(d.hcount / HH, a.nspans, d.batch);
    launch_begin(kKindChunkState, s);
    const cudaError_t le =
        launch_dependent(chunk_state_tc_kernel<N, HH, ONE>, grid, dim3(K::THREADS), K::SMEM, s, tx, tb, a);
    const int r = launch_end(kKindChunkState, s);
    return le != cudaSuccess ? SSD_ERR_CUDA : r;
}

// Multiprocessor count of the current device (cached per device).
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

// A grid that fits one CTA per SM gets the configuration with twice the stages.
template <int N, int HH>
int launch_state_nh(const __nv_bfloat16* x, const __half* B, const StateArgs& a, cudaStream_t s) {
    const int64_t ctas = (int64_t)(a.d.hcount / HH) * a.nspans * a.d.batch;
    if (ctas <= sm_count()) return launch_state_nho<N, HH, true>(x, B, a, s);
    return launch_state_nho<N, HH, false>(x, B, a, s);
}

// Heads per CTA: as many of one group as divide evenly, up to 4 (N <= 128) or 2 (N >= 256); with a
// head range, the CTAs' head blocks must also tile the range and start on a multiple of the block.
template <int N>
int launch_state_n(const __nv_bfloat16* x, const __half* B, const StateArgs& a, cudaStream_t s) {
    switch (chunk_state_heads_per_cta(a.d)) {
        case 4: return launch_state_nh<N, (N <= 128 ? 4 : 2)>(x, B, a, s);
        case 2: return launch_state_nh<N, 2>(x, B, a, s);
        default: return launch_state_nh<N, 1>(x, B, a, s);
    }
}

}  // namespace

int chunk_state_heads_per_cta(const Dims& d) {
    const int hpg = d.nheads / d.ngroups;
    auto fits = [&](int hh) { return hpg % hh == 0 && d.hcount % hh == 0 && d.head0 % hh == 0; };
    const int hmax = (d.dstate <= 128) ? 4 : 2;
    if (hmax >= 4 && fits(4)) return 4;
    if (fits(2)) return 2;
    return 1;
}

int launch_chunk_state_span(const __nv_bfloat16* x, const __half* B, const float* dtt, const float* cs,
                            int span_chunks, const Dims& d, float* S, float* span_decay, const Ctl& ctl,
                            cudaStream_t s, __half* S16) {
    if (span_chunks < 1 || span_chunks > kMaxSpanChunks) return SSD_ERR_UNSUPPORTED;
    StateArgs a;
    a.d = d;
    a.span_chunks = span_chunks;
    a.nspans = ceil_div(d.nchunks, span_chunks);
    a.cs = cs;
    a.dtt = dtt;
    a.S = S;
    a.S16 = S16;
    a.span_decay = span_decay;
    a.ctl = ctl;
    a.rev = 0;
    switch (d.dstate) {
        case 64: return launch_state_n<64>(x, B, a, s);
        case 128: return launch_state_n<128>(x, B, a, s);
        case 256: return launch_state_n<256>(x, B, a, s);
        case 512: return launch_state_n<512>(x, B, a, s);
        default: return SSD_ERR_UNSUPPORTED;
    }
}

int launch_chunk_state_rev(const __nv_bfloat16* dy, const __half* C16, const float* dtt, const float* cs, const Dims& d,
                           float* Z, const Ctl& ctl, cudaStream_t s, __half* Z16) {
    StateArgs a;
    a.d = d;
    a.span_chunks = 1;
    a.nspans = d.nchunks;
    a.cs = cs;
    a.dtt = dtt;
    a.S = Z;
    a.S16 = Z16;
    a.span_decay = nullptr;
    a.ctl = ctl;
    a.rev = 1;
    switch (d.dstate) {
        case 64: return launch_state_n<64>(dy, C16, a, s);
        case 128: return launch_state_n<128>(dy, C16, a, s);
        case 256: return launch_state_n<256>(dy, C16, a, s);
        case 512: return launch_state_n<512>(dy, C16, a, s);
        default: return SSD_ERR_UNSUPPORTED;
    }
}

}  // namespace ssd
