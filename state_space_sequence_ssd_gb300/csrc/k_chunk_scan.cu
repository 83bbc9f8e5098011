// k_chunk_scan.cu -- compute_out on tcgen05 tensor cores, carrying the state
// through 128-token sub-blocks of a span.
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile": three-kernel paragraph
// (compute_out fuses the carried-state term, the decayed causally masked
// interaction matrix and the skip connection into one tiled kernel) and the
// jump-formula paragraph (state advance B^T (w * X) as one matrix product);
// devotd.net page, section 2 (the intermediate matrix stays on chip) and
// section 3 (operand order chosen for the tensor-core input layout, bank
// conflicts avoided -- here by 128-byte swizzled tiles).
//
// One CTA per (head h, span s, batch b).  A span is a run of whole chunks
// that starts from a known state: entry s * state_step of the span-start
// state array (state_step > 1 lets one CTA walk several of the state array's
// spans, carrying the state across their boundaries, so fewer and longer CTAs
// pay the pipeline fill and drain).  The span is walked in sub-blocks of 128
// tokens.  With u_i the in-sub-block inclusive log2
// decay (u_i = log2(e) * sum_{k<=i} dt_k A) and the state h at the
// sub-block start:
//
//   S    : h   <- 2^(u_last) h + B^T (w X),   w_j = 2^(u_last - u_j) dt_j
//   YS   : Yst  = C h                          -> y_i += 2^(u_i) Yst_i
//   CB   : CB   = C B^T                        (128 x 128, f32 in TMEM)
//   mask : M    = CB * 2^(u_i - u_j) dt_j [j <= i] + D [j == i]   (float16, back into TMEM)
//   MX   : Y    = M X                          (A operand read from TMEM; includes the D skip)
//   DX   : Y   += X diag(D)                    (only with one skip weight per channel: D is
//                                               (H, P); X as a K-major A operand, diag(D) a
//                                               float16 64 x 64 tile built once per CTA)
//   y_i  = Y_i + 2^(u_i) Yst_i
//
// The mask never exponentiates more than a 32 x 32 diagonal block per row:
// for a column block q strictly below the row's block, with r the block's
// last position, 2^(u_i - u_j) = 2^(u_i - u_r) * 2^(u_r - u_j), both factors
// <= 1 (u is non-increasing), so no factor overflows.
//
// Roles (480 threads):
//   warps 0-3   mask warpgroup: CB -> M (one row per thread)
//   warps 4-7   state warpgroup: u/dt/column weights of each sub-block, the
//               x tile converted to float16 in place with X' = w X, the
//               float16 copy of the state for C h and the decay of the state
//               held in TMEM
//   warps 8-11  epilogue warpgroup: y = Y + 2^u Yst, each thread storing its
//               128-byte row of y straight from registers; with the z gate
//               it multiplies by z sigmoid(z), the thread's z row loaded into
//               registers one sub-block ahead
//   warp 12     producer of the x tiles and dA_cumsum/dt rows (TMA)
//   warp 13     TMEM owner and single-thread MMA issuer
//   warp 14     producer of the C and B tiles (TMA), running ahead independently
// The MMA issuer polls readiness and issues whichever is ready: the "front"
// of the next sub-block (S, YS, CB) or the M X of a finished mask, keeping at
// most two sub-blocks in flight over two TMEM buffer sets {CB/M/Y, Yst}.  The
// x tile is released as soon as its M X retires.
//
// Precision: all four products run in float16 (kind::f16, f32 accumulate).
// B and C are exact float16 copies of the inputs; the x tile is converted to
// float16 in place (exact for normal-range bfloat16); the derived operands M,
// h and w x are rounded once to float16 (11 significant bits), which keeps
// every output within 1e-2 + 1e-2 |y| where bfloat16 operands do not.
//
// Every wait is bounded (1 s); a role that gives up sets the CTA abort flag
// and the device error word, and all roles fall through to teardown.
#include "common.cuh"
#include "sm100.cuh"
#include "tmap.cuh"
#include "scan_util.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kThreads = 480;
constexpr int kTile = 16384;  // 128 rows x 128 B
constexpr int kWarpTma = 12, kWarpMma = 13, kWarpTmaBC = 14;

template <int N, bool OPT>
struct Cfg {
    static constexpr int NB = N < 128 ? N : 128;  // state rows per n-block
    static constexpr int NBLK = N / NB;
    static constexpr int BOXES = NB / 64;        // 64-column TMA boxes per n-block
    static constexpr int NST = 2;
    static constexpr bool S_FIRST = NBLK <= NST;  // all n-blocks resident: issue every S before YS/CB
    static constexpr int NBUF = (N == 512) ? 1 : 2;
    static constexpr int NX = (N >= 256) ? 2 : 3;  // x tiles in flight
    // RING (N = 512): the float16 copy of the state for C h lives in two 128-row slots, n-block nb
    // in slot nb % 2, instead of all N rows at once; the shared memory this frees holds a second
    // C/B stage, so an n-block's tiles load while the previous n-block's products run.
    static constexpr bool RING = (N == 512);
    static constexpr int SZ_HS = NB * 128;  // one slot
    // TMEM columns
    static constexpr int T_H = 0;
    static constexpr int HC = NBLK * 64;
    static constexpr int T_SET = HC;  // set k at T_SET + k * SET: [CB/M, Y in cols 64..127][Yst]
    static constexpr int SET = 192;
    static constexpr int TCOLS = 512;
    static_assert(HC + NBUF * SET <= TCOLS, "TMEM budget");
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int OFF_X = 0;  // NX x tiles
    static constexpr int OFF_XS = OFF_X + NX * kTile;
    static constexpr int OFF_H = OFF_XS + kTile;
    static constexpr int SZ_H = RING ? 2 * SZ_HS : N * 128;
    static constexpr int OFF_BC = OFF_H + SZ_H;
    static constexpr int SZ_C = BOXES * kTile;
    static constexpr int SZ_STAGE = 2 * SZ_C;  // C then B
    static constexpr int OFF_ZERO = OFF_BC + NST * SZ_STAGE;
    static constexpr int SZ_ZERO = (N == 64) ? kTile : 0;
    static constexpr int OFF_U = OFF_ZERO + SZ_ZERO;  // 3 x {u[128], dt[128], bcol[128], -[128]}
    static constexpr int OFF_CD = OFF_U + 3 * 2048;   // NX x {cs[128], dt[128]} rows, bulk-copied with x
    static constexpr int OFF_DG = OFF_CD + NX * 1024;  // diag(D) 64 x 64 float16, K-major, 128B-swizzled
    static constexpr int OFF_BAR = OFF_DG + (OPT ? 8192 : 0);
    static constexpr int SMEM = OFF_BAR + 512 + 1024;  // + alignment slack
    static_assert(SMEM <= 232448, "shared memory budget");
};

constexpr uint32_t kIdescCB = idesc_fp16(128, 128, false, false);
constexpr uint32_t kIdescYS = idesc_fp16(128, 64, false, true);
constexpr uint32_t kIdescS = idesc_fp16(128, 64, true, true);
constexpr uint32_t kIdescMX = idesc_fp16(128, 64, false, true);
constexpr uint32_t kIdescDX = idesc_fp16(128, 64, false, false);

struct ScanArgs {
    Dims d;
    int span_chunks;  // chunks per span
    int nspans;
    int state_step;    // span-start state of span s: entry s * state_step of the state array
    int state_spans;   // entries per (batch) row of the state array
    const float* cs;    // (b, hcount, nc, Q)
    const float* dtt;   // (b, hcount, nc, Q)
    const float* D;     // (H) or null: the skip term on M's diagonal
    const float* init;  // (b, state_spans, hcount, P, N) span-start states
    __nv_bfloat16* y;   // (b, L, H, P)
    int y32;            // y is 32-byte aligned: rows are stored in 32-byte pieces
    int z32;            // the gate z is 32-byte aligned: rows are loaded in 32-byte pieces
    Ctl ctl;            // error words, wait limit, stall hook
    OutOpts oo;  // D per channel (then D is null: no diagonal skip) and the z gate
};

struct Bars {
    uint64_t x_full[3], x_empty[3];
    uint64_t bc_full[2], bc_empty[2];
    uint64_t uv_ready[3], u_free[3];
    uint64_t cb_full[2], m_ready[2], y_full[2], y_free[2];
    uint64_t xs_ready, xs_free, h_ready, state_done, final_mma;
    uint64_t hs_ready[2], hs_free[2];  // RING: state-copy slot k filled (128 arrivals) / read by C h
    uint64_t stall;                    // never completed: the test hook's wait runs out on it
};

static_assert(sizeof(Bars) <= 512, "barriers fit their shared-memory slot");

// Eight consecutive channels of one output row times z sigmoid(z); zq holds the row's eight bf16 gate values.
__device__ __forceinline__ void gate8(float (&o)[8], const uint4& zq) {
    const uint32_t* zw = reinterpret_cast<const uint32_t*>(&zq);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = zw[i >> 1];
        o[i] *= silu(__uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16)));
    }
}

// OPT: the layer's output options (D per channel, z gate) are compiled in; the plain
// instantiation carries none of their code, registers or shared memory.
template <int N, bool OPT>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                         const __grid_constant__ CUtensorMap tm_C, ScanArgs a) {
    using K = Cfg<N, OPT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars* bar = reinterpret_cast<Bars*>(smem + K::OFF_BAR);
    float* sU = reinterpret_cast<float*>(smem + K::OFF_U);  // buffer k at k*512: u, dt, bcol
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const Dims& d = a.d;
    // hl: local head (the call's intermediates); h = head0 + hl: its head in x, y, z, D and B / C
    const int hl = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int H = d.nheads, HC = d.hcount, G = d.ngroups, Q = d.chunk_size;
    const int h = d.head0 + hl;
    const int g = h / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ts = (int64_t)s * a.span_chunks * Q;
    const int64_t te = min((int64_t)d.seqlen, ts + (int64_t)a.span_chunks * Q);
    const int nsb = (int)((te - ts + 127) / 128);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) {
            mbar_init(&bar->x_full[i], 1);
            mbar_init(&bar->x_empty[i], 1);   // the M X product that read the tile has retired
            mbar_init(&bar->uv_ready[i], 128);
            mbar_init(&bar->u_free[i], 256);  // mask and epilogue are done with this u buffer
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->bc_full[i], 1);
            mbar_init(&bar->bc_empty[i], 1);
            mbar_init(&bar->cb_full[i], 1);
            mbar_init(&bar->m_ready[i], 128);
            mbar_init(&bar->y_full[i], 1);
            mbar_init(&bar->y_free[i], 128);
        }
        mbar_init(&bar->xs_ready, 128);
        mbar_init(&bar->xs_free, 1);
        mbar_init(&bar->h_ready, 128);
        mbar_init(&bar->state_done, 1);
        mbar_init(&bar->final_mma, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->hs_ready[i], 128);
            mbar_init(&bar->hs_free[i], 1);
        }
        mbar_init(&bar->stall, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    int* const err = a.ctl.err;
    const uint64_t wait_ns = a.ctl.wait_ns;
    if (K::SZ_ZERO > 0) {  // rows that pad the state-update A operand to 128 (N = 64)
        uint4* z = reinterpret_cast<uint4*>(smem + K::OFF_ZERO);
        for (int i = threadIdx.x; i < K::SZ_ZERO / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (OPT && a.oo.Dp != nullptr) {
        float dmx = 0.f;
        // diag(D[h, :]) as the B operand of DX: row n (output channel) holds D[h][n] at column k = n.
        // 128B swizzle: row n at (n / 8) * 1024 + (n % 8) * 128, 16-byte chunk j stored at chunk j ^ (n % 8).
        for (int c = threadIdx.x; c < 512; c += kThreads) {
            const int n = (c >> 6) * 8 + ((c >> 3) & 7);
            const int j = (c & 7) ^ (n & 7);  // logical chunk: columns 8j .. 8j+7
            uint32_t v = 0u;  // the diagonal element, placed in its 32-bit word of the chunk
            if (j == (n >> 3)) {
                const float df = a.oo.Dp[h * 64 + n];
                dmx = fmaxf(dmx, fabsf(df));
                const __half dv = __float2half_rn(df);
                const uint32_t bits = *reinterpret_cast<const uint16_t*>(&dv);
                v = (n & 1) ? (bits << 16) : bits;
            }
            const int wi = (n & 7) >> 1;
            reinterpret_cast<uint4*>(smem + K::OFF_DG)[c] =
                make_uint4(wi == 0 ? v : 0u, wi == 1 ? v : 0u, wi == 2 ? v : 0u, wi == 3 ? v : 0u);
        }
        fence_proxy_async_smem();
        flag_f16_range(err, dmx);
    }
    if (warp == kWarpMma) {
        tmem_alloc(&tmem_base_sh, K::TCOLS);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_B);
        tma_prefetch_desc(&tm_C);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dep_wait();  // states, dA_cumsum, dt and the float16 B / C come from earlier launches
    const uint32_t tm = tmem_base_sh;
    volatile int* abort_flag = &abort_sh;

    if (warp == kWarpTma) {
        // ------------------------------------------------------ x / dA_cumsum / dt producer
        if (lane == 0) {
            if (a.ctl.stall) wait_bounded<!OPT>(&bar->stall, 0, abort_flag, err, 30, wait_ns);
            int nissued = 0;  // loads issued; buffer i took those with index % NX == i
            const int64_t rowlen = (int64_t)d.nchunks * Q;
            for (int sb = 0; sb < nsb && !*abort_flag; ++sb) {
                const int t0 = (int)(ts + sb * 128);
                const int xb = sb % K::NX;
                if (!wait_bounded<!OPT>(&bar->x_empty[xb], ((sb / K::NX) & 1) ^ 1, abort_flag, err, 1, wait_ns))
                    break;
                // this sub-block's rows of dA_cumsum and dt (contiguous per (b, h); at most 128)
                const uint32_t cdb = (uint32_t)min((int64_t)128, rowlen - t0) * 4u;
                float* scd = reinterpret_cast<float*>(smem + K::OFF_CD + xb * 1024);
                mbar_arrive_expect_tx(&bar->x_full[xb], kTile + 2 * cdb);
                tma_load_4d(smem + K::OFF_X + xb * kTile, &tm_x, &bar->x_full[xb], 0, h, t0, b);
                bulk_load(scd, a.cs + ((int64_t)b * HC + hl) * rowlen + t0, cdb, &bar->x_full[xb]);
                bulk_load(scd + 128, a.dtt + ((int64_t)b * HC + hl) * rowlen + t0, cdb, &bar->x_full[xb]);
                ++nissued;
            }
            // no load may still be landing in shared memory at teardown
#pragma unroll
            for (int i = 0; i < K::NX; ++i) {
                const int issued = (nissued + K::NX - 1 - i) / K::NX;
                if (issued > 0) mbar_wait_drain(&bar->x_full[i], (issued - 1) & 1, err, 103, kDrainNs);
            }
        }
    } else if (warp == kWarpTmaBC) {
        // ------------------------------------------------------ C / B producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            int nissued = 0;  // stage loads issued; stage i took those with index % NST == i
            for (int sb = 0; sb < nsb && ok && !*abort_flag; ++sb) {
                const int t0 = (int)(ts + sb * 128);
                for (int nb = 0; nb < K::NBLK && ok; ++nb, ++it) {
                    const int st = it % K::NST;
                    ok = wait_bounded<!OPT>(&bar->bc_empty[st], ((it / K::NST) & 1) ^ 1, abort_flag, err, 2,
                                           wait_ns);
                    if (!ok) break;
                    uint8_t* sC = smem + K::OFF_BC + st * K::SZ_STAGE;
                    uint8_t* sB = sC + K::SZ_C;
                    mbar_arrive_expect_tx(&bar->bc_full[st], K::SZ_STAGE);
#pragma unroll
                    for (int bx = 0; bx < K::BOXES; ++bx) {
                        tma_load_4d(sC + bx * kTile, &tm_C, &bar->bc_full[st], nb * K::NB + bx * 64, g, t0, b);
                        tma_load_4d(sB + bx * kTile, &tm_B, &bar->bc_full[st], nb * K::NB + bx * 64, g, t0, b);
                    }
                    ++nissued;
                }
            }
#pragma unroll
            for (int i = 0; i < K::NST; ++i) {
                const int issued = (nissued + K::NST - 1 - i) / K::NST;
                if (issued > 0) mbar_wait_drain(&bar->bc_full[i], (issued - 1) & 1, err, 104, kDrainNs);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sXs = smem_u32(smem + K::OFF_XS);
            const uint32_t sZero = smem_u32(smem + K::OFF_ZERO);
            const uint32_t sH = smem_u32(smem + K::OFF_H);
            const uint32_t sDg = smem_u32(smem + K::OFF_DG);
            const bool dx = OPT && a.oo.Dp != nullptr;
            auto stage_c = [&](int st) -> uint32_t { return smem_u32(smem + K::OFF_BC + st * K::SZ_STAGE); };
            // h[nb] += B_nb^T X'  (K = tokens; A MN-major over two 64-row n boxes)
            auto issue_s = [&](int nb, uint32_t sB) {
                const uint32_t lbo = (K::BOXES == 2) ? (uint32_t)kTile : (sZero - sB);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tm + K::T_H + nb * 64, desc_sw128(sB + kk * 2048, lbo, 1024),
                           desc_sw128(sXs + kk * 2048, 16, 1024), kIdescS, 1);
            };
            // Yst += C_nb h_nb   (K = n, 16 per step); h_nb in its ring slot (RING) or at rows nb NB
            auto issue_ys = [&](int nb, uint32_t set, uint32_t sC) {
                const uint32_t hb = K::RING ? sH + (uint32_t)((nb & 1) * K::SZ_HS) : sH + (uint32_t)(nb * K::NB * 128);
#pragma unroll
                for (int kk = 0; kk < K::NB / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    mma_ss(set + 128, desc_sw128(sC + off, 16, 1024), desc_sw128(hb + kk * 16 * 128, 16, 1024),
                           kIdescYS, (nb | kk) != 0);
                }
            };
            // CB += C_nb B_nb^T   (K = n, 16 per step)
            auto issue_cb = [&](int nb, uint32_t set, uint32_t sC, uint32_t sB) {
#pragma unroll
                for (int kk = 0; kk < K::NB / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    mma_ss(set, desc_sw128(sC + off, 16, 1024), desc_sw128(sB + off, 16, 1024), kIdescCB,
                           (nb | kk) != 0);
                }
            };
            // Y = M X for sub-block q (A = M from TMEM, B = the float16 x tile, MN-major)
            auto issue_mx = [&](int q) {
                const int k = q % K::NBUF;
                const uint32_t sX = smem_u32(smem + K::OFF_X + (q % K::NX) * kTile);
                const uint32_t set = tm + K::T_SET + k * K::SET;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(set + 64, set + kk * 8, desc_sw128(sX + kk * 2048, 16, 1024), kIdescMX, kk > 0);
                if (dx) {  // Y += X diag(D): the same tile read as a K-major A operand (K = channels)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(set + 64, desc_sw128(sX + kk * 32, 16, 1024), desc_sw128(sDg + kk * 32, 16, 1024),
                               kIdescDX, 1);
                }
                mma_commit(&bar->y_full[k]);
                mma_commit(&bar->x_empty[q % K::NX]);
            };
            // front(f): S (state update), then C h, then C B^T; false on a failed wait
            int it = 0;
            int f = 0, m = 0;  // next front to issue, next M X to issue
            // a finished mask's M X goes ahead of the rest of a front (the tensor pipe runs
            // instructions in issue order, and the epilogue and the next front wait on it);
            // measured on GB300 to pay off for N >= 256 (two n-blocks per front) only
            auto mx_if_ready = [&](int f) {
                if (N >= 256 && m < f && mbar_test_wait(&bar->m_ready[m % K::NBUF], (m / K::NBUF) & 1)) {
                    tc_fence_after();
                    issue_mx(m++);
                }
            };
            auto issue_front = [&](int f) -> bool {
                const bool need_S = f + 1 < nsb;
                const int k = f % K::NBUF;
                const uint32_t set = tm + K::T_SET + k * K::SET;
                if (K::S_FIRST) {
                    if (need_S)
                        for (int nb = 0; nb < K::NBLK; ++nb) issue_s(nb, stage_c((it + nb) % K::NST) + K::SZ_C);
                    mma_commit(&bar->xs_free);
                    mx_if_ready(f);
                    for (int nb = 0; nb < K::NBLK; ++nb) issue_ys(nb, set, stage_c((it + nb) % K::NST));
                    mma_commit(&bar->state_done);
                    mx_if_ready(f);
                    for (int nb = 0; nb < K::NBLK; ++nb, ++it) {
                        const int st = it % K::NST;
                        issue_cb(nb, set, stage_c(st), stage_c(st) + K::SZ_C);
                        mma_commit(&bar->bc_empty[st]);
                    }
                } else {
                    // n-blocks streamed one stage at a time
                    for (int nb = 0; nb < K::NBLK; ++nb, ++it) {
                        const int st = it % K::NST;
                        const int use = f * (K::NBLK / 2) + nb / 2;  // RING: use index of slot nb % 2
                        if (nb > 0) {
                            if (!wait_bounded<!OPT>(&bar->bc_full[st], (it / K::NST) & 1, abort_flag, err, 8,
                                                   wait_ns))
                                return false;
                            if (K::RING &&
                                !wait_bounded<!OPT>(&bar->hs_ready[nb & 1], use & 1, abort_flag, err, 9, wait_ns))
                                return false;
                            tc_fence_after();
                        }
                        if (need_S) issue_s(nb, stage_c(st) + K::SZ_C);
                        issue_ys(nb, set, stage_c(st));
                        if (K::RING) mma_commit(&bar->hs_free[nb & 1]);
                        issue_cb(nb, set, stage_c(st), stage_c(st) + K::SZ_C);
                        mma_commit(&bar->bc_empty[st]);
                    }
                    mma_commit(&bar->xs_free);
                    mma_commit(&bar->state_done);
                }
                mma_commit(&bar->cb_full[k]);
                return true;
            };
            auto front_ready = [&](int f) -> bool {
                if (!mbar_test_wait(&bar->xs_ready, f & 1)) return false;
                if (K::RING ? !mbar_test_wait(&bar->hs_ready[0], (f * (K::NBLK / 2)) & 1)
                            : !mbar_test_wait(&bar->h_ready, f & 1))
                    return false;
                const int nres = K::S_FIRST ? K::NBLK : 1;  // stages that must be resident to start
                for (int nb = 0; nb < nres; ++nb)
                    if (!mbar_test_wait(&bar->bc_full[(it + nb) % K::NST], ((it + nb) / K::NST) & 1)) return false;
                if (f >= K::NBUF && !mbar_test_wait(&bar->y_free[f % K::NBUF], ((f / K::NBUF) - 1) & 1))
                    return false;
                return true;
            };
            bool ok = true;
            uint64_t last = globaltimer_ns();
            while (m < nsb && ok) {
                bool did = false;
                if (m < f && mbar_test_wait(&bar->m_ready[m % K::NBUF], (m / K::NBUF) & 1)) {
                    tc_fence_after();
                    issue_mx(m++);
                    did = true;
                } else if (f < nsb && f - m < K::NBUF && front_ready(f)) {
                    tc_fence_after();
                    ok = issue_front(f++);
                    did = true;
                }
                if (did) {
                    last = globaltimer_ns();
                } else {
                    __nanosleep(32);  // leave the issue slots to the math warps sharing this scheduler
                    if (*abort_flag) break;
                    if (globaltimer_ns() - last > wait_ns) {
                        *abort_flag = 1;
                        atomicExch(err, 4);
                        break;
                    }
                }
            }
            // every MMA retired before TMEM is released
            mma_commit(&bar->final_mma);
            mbar_wait_drain(&bar->final_mma, 0, err, 110, kDrainNs);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------ mask warpgroup: CB -> M
        const int r = threadIdx.x;  // TMEM lane == row
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float Dh = (a.D != nullptr) ? a.D[h] : 0.f;  // the skip term rides on M's diagonal
        __half2 mx = __floats2half2_rn(0.f, 0.f);  // largest |M| after rounding to float16 (range flag)
        for (int sb = 0; sb < nsb; ++sb) {
            const int k = sb % K::NBUF;
            const int ub = sb % 3;
            bool ok = wait_bounded<!OPT>(&bar->uv_ready[ub], (sb / 3) & 1, abort_flag, err, 11, wait_ns) &&
                      wait_bounded<!OPT>(&bar->cb_full[k], (sb / K::NBUF) & 1, abort_flag, err, 12, wait_ns);
            ok = __all_sync(0xffffffffu, ok);  // TMEM loads/stores below are warp-collective
            if (!ok) break;
            tc_fence_after();
            const float* su = sU + ub * 512;
            const float* sdt = su + 128;
            const float* sbc = su + 256;
            const float ui = su[r];
            const uint32_t set = tm + lane_base + K::T_SET + k * K::SET;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t o[16];
                if (q > warp) {  // above the diagonal
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = 0u;
                } else {
                    uint32_t v[32];
                    tmem_ld32(set + q * 32, v);
                    tmem_ld_wait(v);
                    const float ue = su[q * 32 + 31];  // u at the block end (its last valid position)
                    const bool diag = q == warp;
                    float m[32];
                    if (!diag || su[q * 32] - ue < 60.f) {
                        // 2^(u_i - u_j) = 2^(u_i - u_e) 2^(u_e - u_j): below the diagonal both factors are <= 1;
                        // on it the block decays by less than 2^60, so the row factor is in [1, 2^60] and
                        // the column weights in [2^-60, 1] dt_j (a warp-uniform branch)
                        const float ar = diag ? fast_exp2(ui - ue) : fast_exp2(fminf(ui - ue, 0.f));
                        float4 bc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) bc[i] = *reinterpret_cast<const float4*>(sbc + q * 32 + 4 * i);
                        const float2 ar2 = make_float2(ar, ar);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {  // packed pairs: half the multiply instructions
                            const float2 w01 = fmul2(ar2, make_float2(bc[i].x, bc[i].y));
                            const float2 w23 = fmul2(ar2, make_float2(bc[i].z, bc[i].w));
                            const float2 m01 = fmul2(make_float2(__uint_as_float(v[4 * i + 0]), __uint_as_float(v[4 * i + 1])), w01);
                            const float2 m23 = fmul2(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), w23);
                            m[4 * i + 0] = m01.x;
                            m[4 * i + 1] = m01.y;
                            m[4 * i + 2] = m23.x;
                            m[4 * i + 3] = m23.y;
                        }
                    } else {  // steep decay in the diagonal block: the exact exponent per element
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 uj = *reinterpret_cast<const float4*>(su + q * 32 + 4 * i);
                            const float4 dj = *reinterpret_cast<const float4*>(sdt + q * 32 + 4 * i);
                            m[4 * i + 0] = __uint_as_float(v[4 * i + 0]) * fast_exp2(fminf(ui - uj.x, 0.f)) * dj.x;
                            m[4 * i + 1] = __uint_as_float(v[4 * i + 1]) * fast_exp2(fminf(ui - uj.y, 0.f)) * dj.y;
                            m[4 * i + 2] = __uint_as_float(v[4 * i + 2]) * fast_exp2(fminf(ui - uj.z, 0.f)) * dj.z;
                            m[4 * i + 3] = __uint_as_float(v[4 * i + 3]) * fast_exp2(fminf(ui - uj.w, 0.f)) * dj.w;
                        }
                    }
                    if (diag) {  // causal mask and the skip term D on the diagonal
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) {
                            const int j = q * 32 + jj;
                            m[jj] = (j <= r) ? m[jj] : 0.f;
                            m[jj] += (j == r) ? Dh : 0.f;
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) o[jj] = pack_f16x2(m[2 * jj], m[2 * jj + 1]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) hmax_abs4(mx, o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                }
                tmem_st16(set + q * 16, o);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar->m_ready[k]);
            mbar_arrive(&bar->u_free[ub]);
        }
        flag_f16_range(err, hmax_to_float(mx));
    } else if (warp < 8) {
        // ------------------------------------------------------ state warpgroup
        // A failed wait turns the remaining work into no-ops but keeps every arrival.
        const int r = threadIdx.x - 128;  // TMEM lane (warp % 4 == warp - 4)
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        const int64_t PN = (int64_t)d.headdim * N;
        const float* init = a.init + (((int64_t)b * a.state_spans + (int64_t)s * a.state_step) * HC + hl) * PN;
        bool ok = true;
        __half2 mx = __floats2half2_rn(0.f, 0.f);  // largest |x|, |w x|, |state copy| in float16 (range flag)
        float prev_raw = 0.f;  // raw dA_cumsum of the token before this sub-block (same chunk)
        for (int sb = 0; sb < nsb; ++sb) {
            const int64_t t0 = ts + sb * 128;
            const int nv = (int)min((int64_t)128, te - t0);
            const int xb = sb % K::NX;
            const int ub = sb % 3;
            float* su = sU + ub * 512;
            // 1. u, dt and the factorized column weights of this sub-block, each computed by its
            //    own thread from the dA_cumsum/dt rows that arrived with the x tile
            if (sb >= 3)
                ok = ok && wait_bounded<!OPT>(&bar->u_free[ub], ((sb / 3) - 1) & 1, abort_flag, err, 17, wait_ns);
            ok = ok && wait_bounded<!OPT>(&bar->x_full[xb], (sb / K::NX) & 1, abort_flag, err, 13, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            const float* scs = reinterpret_cast<const float*>(smem + K::OFF_CD + xb * 1024);
            const int p0 = (int)(t0 % Q);
            const float prev = (p0 > 0) ? prev_raw : 0.f;
            const bool valid = r < nv;
            float u = 0.f, ulast = 0.f, dtv = 0.f, bcol = 0.f;
            if (ok) {
                ulast = sub_block_decay(scs, prev, p0, Q, nv - 1);
                if (valid) {
                    u = sub_block_decay(scs, prev, p0, Q, r);
                    dtv = scs[128 + r];
                    // weight for the factorized mask: 2^(u_end - u_r) dt_r, end = last valid
                    // position of r's 32-block
                    const float uend = sub_block_decay(scs, prev, p0, Q, min(r | 31, nv - 1));
                    bcol = fast_exp2(fminf(uend - u, 0.f)) * dtv;
                } else {
                    u = ulast;
                }
                prev_raw = scs[nv - 1];
            }
            su[r] = u;
            su[128 + r] = dtv;
            su[256 + r] = bcol;
            mbar_arrive(&bar->uv_ready[ub]);
            const float dsb = exp2f(ulast);
            // 2. x tile -> float16 in place, and X' = w x into the single X' buffer once the
            //    previous sub-block's state update has read it
            if (sb > 0) ok = ok && wait_bounded<!OPT>(&bar->xs_free, (sb - 1) & 1, abort_flag, err, 14, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                const float w = valid ? fast_exp2(fminf(ulast - u, 0.f)) * dtv : 0.f;
                uint8_t* xrow = smem + K::OFF_X + xb * kTile;
                uint8_t* xsrow = smem + K::OFF_XS;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t off = sw128_offset(r, ch);
                    const uint4 v = *reinterpret_cast<const uint4*>(xrow + off);
                    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v);
                    uint4 xo, wo;
                    uint32_t* x4 = reinterpret_cast<uint32_t*>(&xo);
                    uint32_t* w4 = reinterpret_cast<uint32_t*>(&wo);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 fv = __bfloat1622float2(p2[e]);
                        x4[e] = pack_f16x2(fv.x, fv.y);
                        const float2 fw = fmul2(fv, make_float2(w, w));
                        w4[e] = pack_f16x2(fw.x, fw.y);
                    }
                    hmax_abs4(mx, x4[0], x4[1], x4[2], x4[3]);
                    hmax_abs4(mx, w4[0], w4[1], w4[2], w4[3]);
                    *reinterpret_cast<uint4*>(xrow + off) = xo;
                    *reinterpret_cast<uint4*>(xsrow + off) = wo;
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&bar->xs_ready);
            // 3. state h_sb -> float16 copy for C h, and h <- 2^(u_last) h in TMEM
            if (sb > 0) {
                ok = ok && wait_bounded<!OPT>(&bar->state_done, (sb - 1) & 1, abort_flag, err, 15, wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
            }
            if (ok) {
                uint8_t* hbase = smem + K::OFF_H;
#pragma unroll 1
                for (int nb = 0; nb < K::NBLK; ++nb) {
                    const int n = nb * K::NB + (r % K::NB);
                    const bool real = r < K::NB;  // N = 64: lanes 64..127 are padding
                    float hv[64];
                    if (sb == 0) {
#pragma unroll
                        for (int p = 0; p < 64; ++p) hv[p] = real ? init[(int64_t)p * N + n] : 0.f;
                    } else {
                        uint32_t v[32];
                        tmem_ld32(tm + lane_base + K::T_H + nb * 64, v);
                        tmem_ld_wait(v);
#pragma unroll
                        for (int p = 0; p < 32; ++p) hv[p] = __uint_as_float(v[p]);
                        tmem_ld32(tm + lane_base + K::T_H + nb * 64 + 32, v);
                        tmem_ld_wait(v);
#pragma unroll
                        for (int p = 0; p < 32; ++p) hv[32 + p] = __uint_as_float(v[p]);
                    }
                    if (K::RING) {  // the slot's previous n-block has been read by its C h product
                        const int use = sb * (K::NBLK / 2) + nb / 2;
                        if (use >= 1)
                            ok = wait_bounded<!OPT>(&bar->hs_free[nb & 1], (use - 1) & 1, abort_flag, err, 19,
                                                   wait_ns);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                    }
                    if (real) {
                        // smem row: state index n, or its row in the ring slot
                        const int hr = K::RING ? r : nb * K::NB + r;
                        uint8_t* hdst = K::RING ? hbase + (nb & 1) * K::SZ_HS : hbase;
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            uint4 v;
                            v.x = pack_f16x2(hv[ch * 8 + 0], hv[ch * 8 + 1]);
                            v.y = pack_f16x2(hv[ch * 8 + 2], hv[ch * 8 + 3]);
                            v.z = pack_f16x2(hv[ch * 8 + 4], hv[ch * 8 + 5]);
                            v.w = pack_f16x2(hv[ch * 8 + 6], hv[ch * 8 + 7]);
                            hmax_abs4(mx, v.x, v.y, v.z, v.w);
                            *reinterpret_cast<uint4*>(hdst + sw128_offset(hr, ch)) = v;
                        }
                    }
                    uint32_t o[16];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                        for (int p = 0; p < 16; p += 2) {  // packed pairs
                            const float2 f = fmul2(make_float2(hv[q4 * 16 + p], hv[q4 * 16 + p + 1]), make_float2(dsb, dsb));
                            o[p] = __float_as_uint(f.x);
                            o[p + 1] = __float_as_uint(f.y);
                        }
                        tmem_st16(tm + lane_base + K::T_H + nb * 64 + q4 * 16, o);
                    }
                    if (K::RING) {  // this n-block's copy and decayed state are ready for S, C h
                        tmem_st_wait();
                        fence_proxy_async_smem();
                        tc_fence_before();
                        mbar_arrive(&bar->hs_ready[nb & 1]);
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
            }
            mbar_arrive(&bar->h_ready);
        }
        flag_f16_range(err, hmax_to_float(mx));
    } else if (warp < 12) {
        // ------------------------------------------------------ epilogue warpgroup
        const int r = threadIdx.x - 256;  // TMEM lane (warp % 4 == warp - 8)
        const uint32_t lane_base = (uint32_t)((warp - 8) * 32) << 16;
        const bool gate = OPT && a.oo.z != nullptr;  // uniform over the CTA
        uint4 zq[8];                                 // this thread's z row of the coming sub-block
        if (gate && r < min((int64_t)128, te - ts)) {
            const uint4* zr = reinterpret_cast<const uint4*>(a.oo.z + (((int64_t)b * d.seqlen + ts + r) * H + h) * 64);
            load_z_row(zr, a.z32, zq);
        }
        bool ok = true;
        for (int sb = 0; sb < nsb; ++sb) {
            const int64_t t0 = ts + sb * 128;
            const int nv = (int)min((int64_t)128, te - t0);
            const int k = sb % K::NBUF;
            const int ub = sb % 3;
            ok = ok && wait_bounded<!OPT>(&bar->y_full[k], (sb / K::NBUF) & 1, abort_flag, err, 16, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            const float e = fast_exp2(fminf(sU[ub * 512 + r], 0.f));
            mbar_arrive(&bar->u_free[ub]);
            if (ok) {
                const uint32_t set = tm + lane_base + K::T_SET + k * K::SET;
                const int64_t row = (((int64_t)b * d.seqlen + t0 + r) * H + h) * 64;
                uint4* yrow = reinterpret_cast<uint4*>(a.y + row);
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    uint32_t yv[32], sv[32];
                    tmem_ld32(set + 64 + half * 32, yv);
                    tmem_ld32(set + 128 + half * 32, sv);
                    tmem_ld_wait(sv);
                    tmem_ld_wait(yv);
                    if (half == 1) {
                        tc_fence_before();
                        mbar_arrive(&bar->y_free[k]);  // this TMEM set may be reused
                    }
                    if (r < nv) {
                        uint4 ov[4];  // this half-row, bfloat16
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            float o[8];
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {  // packed pairs
                                const float2 f = ffma2(make_float2(e, e),
                                                       make_float2(__uint_as_float(sv[ch * 8 + i]), __uint_as_float(sv[ch * 8 + i + 1])),
                                                       make_float2(__uint_as_float(yv[ch * 8 + i]), __uint_as_float(yv[ch * 8 + i + 1])));
                                o[i] = f.x;
                                o[i + 1] = f.y;
                            }
                            if (gate) gate8(o, zq[ch]);
                            uint32_t* o4 = reinterpret_cast<uint32_t*>(&ov[ch]);
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) o4[e2] = pack_bf16x2(o[2 * e2], o[2 * e2 + 1]);
                        }
                        // every lane writes its own 128-byte row: 32-byte stores halve the store
                        // instructions (and the L1 wavefronts of rows 4 KB apart) against 16-byte ones
                        if (a.y32) {
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2) st_global_32B(yrow + half * 4 + 2 * c2, ov[2 * c2], ov[2 * c2 + 1]);
                        } else {
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch) yrow[half * 4 + ch] = ov[ch];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) zq[i] = zq[i + 4];  // the row's second half moves down
                }
            } else {
                mbar_arrive(&bar->y_free[k]);
            }
            if (gate && t0 + 128 + r < te) {  // the next sub-block's z row, in flight during the next wait
                const uint4* zr =
                    reinterpret_cast<const uint4*>(a.oo.z + (((int64_t)b * d.seqlen + t0 + 128 + r) * H + h) * 64);
                load_z_row(zr, a.z32, zq);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tm, K::TCOLS);
}

template <int N, bool OPT>
int launch_scan_n(const __nv_bfloat16* x, const __half* B, const __half* C, const ScanArgs& a, cudaStream_t s) {
    const Dims& d = a.d;
    CUtensorMap tx, tb, tc;
    const uint64_t dx[4] = {(uint64_t)d.headdim, (uint64_t)d.nheads, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint64_t dbc[4] = {(uint64_t)d.dstate, (uint64_t)d.ngroups, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint32_t box_in[4] = {64, 1, 128, 1};
    if (!make_tmap_16b_4d(&tx, x, dx, box_in) || !make_tmap_16b_4d(&tb, B, dbc, box_in) ||
        !make_tmap_16b_4d(&tc, C, dbc, box_in))
        return SSD_ERR_CUDA;
    const int smem = Cfg<N, OPT>::SMEM;
    if (ensure_smem_limit(reinterpret_cast<const void*>(chunk_scan_tc_kernel<N, OPT>), smem) != SSD_OK)
        return SSD_ERR_CUDA;
    dim3 grid(d.hcount, a.nspans, d.batch);
    launch_begin(kKindChunkScan, s);
    const cudaError_t le = launch_dependent(chunk_scan_tc_kernel<N, OPT>, grid, dim3(kThreads), smem, s, tx, tb, tc, a);
    const int r = launch_end(kKindChunkScan, s);
    return le != cudaSuccess ? SSD_ERR_CUDA : r;
}

}  // namespace

int launch_chunk_scan_span(const __nv_bfloat16* x, const __half* B, const __half* C, const float* dtt,
                           const float* cs, const float* D, const float* span_states, int span_chunks, const Dims& d,
                           __nv_bfloat16* y, const Ctl& ctl, cudaStream_t s, const OutOpts& oo, int state_step) {
    if (chunk_scan_pair_supported(d, oo))
        return launch_chunk_scan_pair(x, B, C, dtt, cs, D, span_states, span_chunks, d, y, ctl, s, state_step);
    ScanArgs a;
    a.d = d;
    a.span_chunks = span_chunks * state_step;
    a.nspans = ceil_div(d.nchunks, a.span_chunks);
    a.state_step = state_step;
    a.state_spans = ceil_div(d.nchunks, span_chunks);
    a.cs = cs;
    a.dtt = dtt;
    a.D = D;
    a.init = span_states;
    a.y = y;
    a.y32 = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
    a.z32 = (reinterpret_cast<uintptr_t>(oo.z) & 31u) == 0;
    a.ctl = ctl;
    a.oo = oo;
    if (oo.Dp != nullptr) a.D = nullptr;  // the skip moves from M's diagonal to the X diag(D) product
    const bool opt = oo.Dp != nullptr || oo.z != nullptr;
    switch (d.dstate) {
        case 64: return opt ? launch_scan_n<64, true>(x, B, C, a, s) : launch_scan_n<64, false>(x, B, C, a, s);
        case 128: return opt ? launch_scan_n<128, true>(x, B, C, a, s) : launch_scan_n<128, false>(x, B, C, a, s);
        case 256: return opt ? launch_scan_n<256, true>(x, B, C, a, s) : launch_scan_n<256, false>(x, B, C, a, s);
        case 512: return opt ? launch_scan_n<512, true>(x, B, C, a, s) : launch_scan_n<512, false>(x, B, C, a, s);
        default: return SSD_ERR_UNSUPPORTED;
    }
}

}  // namespace ssd
