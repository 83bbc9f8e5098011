// k_chunk_scan_pair.cu -- compute_out for two heads of one B/C group per CTA, in
// lockstep, on tcgen05 tensor cores (state sizes 64 and 128).
//
// disconfirmai.com page "Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile": three-kernel paragraph (compute_out
// fuses the carried-state term, the decayed causally masked interaction matrix
// and the skip connection) and jump-formula paragraph (the state advance over
// a run of tokens is one product B^T (w X)); devotd.net page, section 2 (the
// intermediate matrix stays on chip) and section 3 (operand order chosen for
// the tensor-core input layout, 128-byte swizzled tiles against bank
// conflicts).
//
// The two heads h0, h0 + 1 of a CTA share their group's B and C, so one load
// of each B/C tile and one C B^T serve both, and the state products are one
// MMA of width 2 x 64.  Per 128-token sub-block, with u the in-sub-block
// inclusive log2 decay of each head (u_i = log2(e) sum_{k<=i} dt_k A) and the
// state at the sub-block start held TRANSPOSED in TMEM, lane (head, p),
// column n (the layout of the state in memory, (P, N) per head):
//
//   S   hT  <- 2^(u_last) hT + X'^T B        X'_j = w_j x_j, w_j = 2^(u_last - u_j) dt_j
//                                            (M = 128 = both heads' p, N = dstate, K = tokens)
//   CB  CB   = C B^T                         (128 x 128, once for both heads)
//   YS  Yst  = C H^T                         (H = float16 copy of hT; N = both heads' p)
//   mask M_h = CB * 2^(u_i - u_j) dt_j [j <= i]   (float16, in place over CB)
//   MX  Y_h  = M_h X_h + X_h diag(D_h)       (A from TMEM; the skip term as one more small product on a
//                                            float16 diag(D_h) tile built once per CTA)
//   y_i = Y_i + 2^(u_i) Yst_i
//
// Roles (736 threads):
//   warps 0-7   mask, two warpgroups MG = 0, 1, warpgroup MG taking 32-column
//               blocks 2 MG and 2 MG + 1 of every row of CB (one row per
//               thread); the two heads' masked rows are written back into the
//               row's own CB columns, interleaved per 16-column half-block (M_0
//               of its 16 positions in 8 packed columns, then M_1), so every
//               half is read before it is overwritten
//   warps 8-15  state, two warpgroups SX = 0, 1 (the serial chain of the pass,
//               split in halves): per sub-block (a) the decays of head SX for
//               the thread's token row, (b) the float16 copy H of half SX of
//               the columns of the state row (head, p) of the thread and their
//               decay in TMEM, (c) X' = w x written over the bf16 x tile of head
//               SX (the x row kept in registers), (d) once S has read X', the
//               float16 x row written in its place for M X
//   warps 16-19 epilogue: y = Y + 2^u Yst for both heads, each thread storing
//               its two 128-byte rows of y
//   warp 20     x / dA_cumsum / dt producer (TMA and bulk copies)
//   warp 21     TMEM owner and single-thread MMA issuer, in order per sub-block
//               (C B^T first, then S, C H^T, the skip term X diag(D) and M X)
//   warp 22     B / C producer: a ring of three tile slots (B of sub-block k,
//               C of k, B of k + 1, ...); B is released after S and C B^T, C
//               after YS, so two sub-blocks' tiles are in flight in three slots
// TMEM: hT [0, 128) | CB / M [128, 256) | Yst [256, 384) | Y [384, 512).
//
// Precision as in k_chunk_scan.cu: float16 operands (B, C exact copies; x exact;
// X', H and M rounded once), f32 accumulation; a value outside float16's finite
// range raises the range flag.  Every wait is bounded; a role that gives up
// sets the CTA abort flag and the error word, and all roles fall through to a
// teardown that lets issued copies and products finish.
#include "common.cuh"
#include "sm100.cuh"
#include "tmap.cuh"
#include "scan_util.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kThreads = 736;
constexpr int kTile = 16384;  // 128 rows x 128 B
constexpr int kWarpTma = 20, kWarpMma = 21, kWarpTmaBC = 22;

template <int N>
struct PCfg {
    static_assert(N == 64 || N == 128, "the paired kernel covers state sizes 64 and 128");
    static constexpr int NBOX = N / 64;           // 64-column boxes per B / C tile and K-blocks of H
    static constexpr int SLOT = NBOX * kTile;     // one B or C tile
    static constexpr int NSLOT = (N == 64) ? 4 : 3;
    static constexpr int NX = (N == 64) ? 3 : 2;  // x stages (two heads each)
    // TMEM columns
    static constexpr int T_H = 0, T_CB = 128, T_YS = 256, T_Y = 384, TCOLS = 512;
    // shared memory (offsets from a 1024-aligned base)
    static constexpr int OFF_X = 0;                         // stage s, head hh at (2 s + hh) kTile
    static constexpr int OFF_H = OFF_X + NX * 2 * kTile;    // K-major rows (head, p), NBOX K-blocks of 64 n
    static constexpr int OFF_BC = OFF_H + NBOX * kTile;     // NSLOT tile slots
    static constexpr int OFF_U = OFF_BC + NSLOT * SLOT;     // 3 x 2 heads x {u, dt, bcol, -}[128] floats
    static constexpr int OFF_CD = OFF_U + 3 * 2 * 2048;     // NX x 2 heads x {cs, dt}[128] floats
    static constexpr int OFF_DG = OFF_CD + NX * 2 * 1024;   // 2 x diag(D_h) 64 x 64 float16, K-major, swizzled
    static constexpr int OFF_BAR = OFF_DG + 2 * 8192;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;       // + alignment slack
    static_assert(SMEM <= 232448, "shared memory budget");
};

constexpr uint32_t kIdescMX = idesc_fp16(128, 64, false, true);
constexpr uint32_t kIdescDX = idesc_fp16(128, 64, false, false);  // X (K-major over channels) diag(D)
constexpr uint32_t kIdescKK = idesc_fp16(128, 128, false, false);  // C B^T and C H^T: both operands K-major

struct PairArgs {
    Dims d;
    int span_chunks;   // chunks per span of this launch
    int nspans;
    int state_step;    // span-start state of span s: entry s * state_step of the state array
    int state_spans;   // entries per (batch) row of the state array
    const float* cs;   // (b, hcount, nc, Q)
    const float* dtt;  // (b, hcount, nc, Q)
    const float* D;    // (H) or null
    const float* init; // (b, state_spans, hcount, P, N) span-start states
    __nv_bfloat16* y;  // (b, L, H, P)
    int y32;           // y is 32-byte aligned: rows are stored in 32-byte pieces
    Ctl ctl;
};

struct PBars {
    uint64_t x_full[3], x_empty[3];
    uint64_t bc_full[4], bc_empty[4];
    uint64_t uv_ready[3], u_free[3];
    uint64_t xs_ready, s_done, h_ready, ys_done, xf_ready, cb_full, m_ready, y_full, y_free;
    uint64_t final_mma, stall;
};
static_assert(sizeof(PBars) <= 512, "barriers fit their shared-memory slot");

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_pair_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                           const __grid_constant__ CUtensorMap tm_C, PairArgs a) {
    using K = PCfg<N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PBars* bar = reinterpret_cast<PBars*>(smem + K::OFF_BAR);
    float* sU = reinterpret_cast<float*>(smem + K::OFF_U);  // buffer ub, head hh at (2 ub + hh) * 512
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const Dims& d = a.d;
    // hl0: first local head (the call's intermediates); h0 = head0 + hl0: its head in x, y, D and B / C
    const int hl0 = 2 * blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int H = d.nheads, HC = d.hcount, G = d.ngroups, Q = d.chunk_size;
    const int h0 = d.head0 + hl0;
    const int g = h0 / (H / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ts = (int64_t)s * a.span_chunks * Q;
    const int64_t te = min((int64_t)d.seqlen, ts + (int64_t)a.span_chunks * Q);
    const int nsb = (int)((te - ts + 127) / 128);
    const int64_t rowlen = (int64_t)d.nchunks * Q;  // dA_cumsum / dt row length per (b, h)

    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) {
            mbar_init(&bar->x_full[i], 1);
            mbar_init(&bar->x_empty[i], 1);
            mbar_init(&bar->uv_ready[i], 256);
            mbar_init(&bar->u_free[i], 384);  // both mask warpgroups and the epilogue are done with this u buffer
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bar->bc_full[i], 1);
            mbar_init(&bar->bc_empty[i], 1);
        }
        mbar_init(&bar->xs_ready, 256);
        mbar_init(&bar->s_done, 1);
        mbar_init(&bar->h_ready, 256);
        mbar_init(&bar->ys_done, 1);
        mbar_init(&bar->xf_ready, 256);
        mbar_init(&bar->cb_full, 1);
        mbar_init(&bar->m_ready, 256);
        mbar_init(&bar->y_full, 1);
        mbar_init(&bar->y_free, 128);
        mbar_init(&bar->final_mma, 1);
        mbar_init(&bar->stall, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    int* const err = a.ctl.err;
    const uint64_t wait_ns = a.ctl.wait_ns;
    if (a.D != nullptr) {
        // diag(D_h) of each head as the B operand of Y_h += X_h diag(D_h): row n (output channel) holds D_h
        // at column k = n.  128B swizzle: row n at (n / 8) * 1024 + (n % 8) * 128, 16-byte chunk j stored
        // at chunk j ^ (n % 8).
        for (int c = threadIdx.x; c < 1024; c += kThreads) {
            const int hh = c >> 9, cc = c & 511;
            const int n = (cc >> 6) * 8 + ((cc >> 3) & 7);
            const int j = (cc & 7) ^ (n & 7);  // logical chunk: columns 8j .. 8j+7
            uint32_t v = 0u;                   // the diagonal element, placed in its 32-bit word of the chunk
            if (j == (n >> 3)) {
                const __half dv = __float2half_rn(a.D[h0 + hh]);
                const uint32_t bits = *reinterpret_cast<const uint16_t*>(&dv);
                v = (n & 1) ? (bits << 16) : bits;
            }
            const int wi = (n & 7) >> 1;
            reinterpret_cast<uint4*>(smem + K::OFF_DG)[c] =
                make_uint4(wi == 0 ? v : 0u, wi == 1 ? v : 0u, wi == 2 ? v : 0u, wi == 3 ? v : 0u);
        }
        fence_proxy_async_smem();
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
    auto xtile = [&](int stage, int hh) -> uint8_t* { return smem + K::OFF_X + (2 * stage + hh) * kTile; };
    auto slot = [&](int i) -> uint8_t* { return smem + K::OFF_BC + (i % K::NSLOT) * K::SLOT; };

    if (warp == kWarpTma) {
        // ------------------------------------------------------ x / dA_cumsum / dt producer
        if (lane == 0) {
            if (a.ctl.stall) wait_bounded<false>(&bar->stall, 0, abort_flag, err, 30, wait_ns);
            int nissued = 0;
            for (int k = 0; k < nsb && !*abort_flag; ++k) {
                const int xs = k % K::NX;
                if (!wait_bounded<false>(&bar->x_empty[xs], ((k / K::NX) & 1) ^ 1, abort_flag, err, 31, wait_ns))
                    break;
                const int t0 = (int)(ts + (int64_t)k * 128);
                const uint32_t cdb = (uint32_t)min((int64_t)128, rowlen - t0) * 4u;
                mbar_arrive_expect_tx(&bar->x_full[xs], 2 * kTile + 4 * cdb);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float* scd = reinterpret_cast<float*>(smem + K::OFF_CD + (2 * xs + hh) * 1024);
                    const int64_t row = ((int64_t)b * HC + hl0 + hh) * rowlen + t0;
                    tma_load_4d(xtile(xs, hh), &tm_x, &bar->x_full[xs], 0, h0 + hh, t0, b);
                    bulk_load(scd, a.cs + row, cdb, &bar->x_full[xs]);
                    bulk_load(scd + 128, a.dtt + row, cdb, &bar->x_full[xs]);
                }
                ++nissued;
            }
#pragma unroll
            for (int i = 0; i < K::NX; ++i) {  // every issued load has landed before teardown
                const int issued = (nissued + K::NX - 1 - i) / K::NX;
                if (issued > 0) mbar_wait_drain(&bar->x_full[i], (issued - 1) & 1, err, 131, kDrainNs);
            }
        }
    } else if (warp == kWarpTmaBC) {
        // ------------------------------------------------------ B / C producer (ring of tile slots)
        if (lane == 0) {
            int nissued = 0;  // tiles issued: tile i = 2 k + (0: B, 1: C) in slot i % NSLOT
            for (int k = 0; k < nsb && !*abort_flag; ++k) {
                const int t0 = (int)(ts + (int64_t)k * 128);
                bool ok = true;
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    const int i = 2 * k + which;
                    const int sl = i % K::NSLOT;
                    ok = wait_bounded<false>(&bar->bc_empty[sl], ((i / K::NSLOT) & 1) ^ 1, abort_flag, err, 32, wait_ns);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&bar->bc_full[sl], K::SLOT);
#pragma unroll
                    for (int bx = 0; bx < K::NBOX; ++bx)
                        tma_load_4d(slot(i) + bx * kTile, which ? &tm_C : &tm_B, &bar->bc_full[sl], bx * 64, g, t0, b);
                    ++nissued;
                }
                if (!ok) break;
            }
#pragma unroll
            for (int sl = 0; sl < K::NSLOT; ++sl) {
                const int issued = (nissued + K::NSLOT - 1 - sl) / K::NSLOT;
                if (issued > 0) mbar_wait_drain(&bar->bc_full[sl], (issued - 1) & 1, err, 132, kDrainNs);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idescS = idesc_fp16(128, N, true, true);
            const uint32_t sH = smem_u32(smem + K::OFF_H);
            for (int k = 0; k < nsb; ++k) {
                const int iB = 2 * k, iC = 2 * k + 1;
                const uint32_t sB = smem_u32(slot(iB)), sC = smem_u32(slot(iC));
                const uint32_t sX0 = smem_u32(xtile(k % K::NX, 0));
                // CB = C B^T (K = n, 16 per step) first, so that the mask can start while S waits for the
                // state warpgroups; it writes the CB region, which the previous M X read (products run in
                // issue order)
                if (!wait_bounded<false>(&bar->bc_full[iB % K::NSLOT], (iB / K::NSLOT) & 1, abort_flag, err, 35, wait_ns) ||
                    !wait_bounded<false>(&bar->bc_full[iC % K::NSLOT], (iC / K::NSLOT) & 1, abort_flag, err, 36, wait_ns))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    mma_ss(tm + K::T_CB, desc_sw128(sC + off, 16, 1024), desc_sw128(sB + off, 16, 1024), kIdescKK, kk > 0);
                }
                mma_commit(&bar->cb_full);
                // S: hT (+)= X'^T B  -- A = both heads' X' (MN-major, heads kTile apart), B = the B tile (MN-major)
                if (!wait_bounded<false>(&bar->xs_ready, k & 1, abort_flag, err, 33, wait_ns) ||
                    !wait_bounded<false>(&bar->h_ready, k & 1, abort_flag, err, 34, wait_ns))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tm + K::T_H, desc_sw128(sX0 + kk * 2048, kTile, 1024), desc_sw128(sB + kk * 2048, kTile, 1024),
                           idescS, 1);
                mma_commit(&bar->s_done);
                mma_commit(&bar->bc_empty[iB % K::NSLOT]);
                // Yst = C H^T once the epilogue has read the previous sub-block's Y and Yst
                if (k > 0 && !wait_bounded<false>(&bar->y_free, (k - 1) & 1, abort_flag, err, 37, wait_ns)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
                    mma_ss(tm + K::T_YS, desc_sw128(sC + off, 16, 1024), desc_sw128(sH + off, 16, 1024), kIdescKK, kk > 0);
                }
                mma_commit(&bar->ys_done);
                mma_commit(&bar->bc_empty[iC % K::NSLOT]);
                // the skip term first, Y_h = X_h diag(D_h) (the x tile read K-major), as soon as the float16
                // x tile is written: it needs no mask, so it runs while the mask warpgroups work
                if (!wait_bounded<false>(&bar->xf_ready, k & 1, abort_flag, err, 39, wait_ns)) break;
                tc_fence_after();
                const bool skip = a.D != nullptr;
                if (skip) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t sX = smem_u32(xtile(k % K::NX, hh));
                        const uint32_t sDg = smem_u32(smem + K::OFF_DG + hh * 8192);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tm + K::T_Y + 64 * hh, desc_sw128(sX + kk * 32, 16, 1024),
                                   desc_sw128(sDg + kk * 32, 16, 1024), kIdescDX, kk > 0);
                    }
                }
                // Y_h (+)= M_h X_h: A = M_h from TMEM (16-column half hf of block q holds M_0 then M_1 of its 16
                // positions, 8 columns each), B = the float16 x tile of head hh (MN-major)
                if (!wait_bounded<false>(&bar->m_ready, k & 1, abort_flag, err, 38, wait_ns)) break;
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t sX = smem_u32(xtile(k % K::NX, hh));
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tm + K::T_Y + 64 * hh, tm + K::T_CB + 32 * (kk >> 1) + 16 * (kk & 1) + 8 * hh,
                               desc_sw128(sX + kk * 2048, 16, 1024), kIdescMX, skip || kk > 0);
                }
                mma_commit(&bar->y_full);
                mma_commit(&bar->x_empty[k % K::NX]);
            }
            // every product retired before TMEM is released
            mma_commit(&bar->final_mma);
            mbar_wait_drain(&bar->final_mma, 0, err, 140, kDrainNs);
        }
    } else if (warp < 8) {
        // ------------------------------------------------------ mask warpgroups MG = 0, 1: CB -> M_0, M_1
        // Row r; warpgroup MG handles the 32-column blocks q = 2 MG, 2 MG + 1 of the row (the causal
        // triangle gives each warp at most two blocks of work).
        const int r = threadIdx.x & 127;
        const int wq = warp & 3;  // row block of this warp
        const int MG = warp >> 2;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        __half2 mx = __floats2half2_rn(0.f, 0.f);
        for (int k = 0; k < nsb; ++k) {
            const int ub = k % 3;
            bool ok = wait_bounded<false>(&bar->uv_ready[ub], (k / 3) & 1, abort_flag, err, 41, wait_ns) &&
                      wait_bounded<false>(&bar->cb_full, k & 1, abort_flag, err, 42, wait_ns);
            ok = __all_sync(0xffffffffu, ok);  // TMEM loads/stores below are warp-collective
            if (!ok) break;
            tc_fence_after();
            const uint32_t cb = tm + lane_base + K::T_CB;
            float ui[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) ui[hh] = sU[(2 * ub + hh) * 512 + r];
#pragma unroll 1
            for (int q = 2 * MG; q < 2 * MG + 2; ++q) {
                if (q > wq) {  // above the diagonal: both heads' blocks are zero
                    uint32_t z[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) z[e] = 0u;
                    tmem_st32(cb + 32 * q, z);
                    continue;
                }
                // the block in two halves of 16 columns; half hf of CB is read before its 16 columns receive
                // M_0 then M_1 of the same 16 positions (8 packed columns each)
                const float* su0 = sU + (2 * ub) * 512;
                const float* su1 = su0 + 512;
                const bool diag = q == wq;
                bool fact[2] = {true, true};  // diagonal block: factorized when its decay is below 2^60
                float ar[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float* su = hh ? su1 : su0;
                    const float uih = hh ? ui[1] : ui[0];  // selects: no local-memory array
                    const float ue = su[q * 32 + 31];       // u at the block end (its last valid position)
                    if (diag) {
                        // the block decays by less than 2^60: 2^(u_i - u_j) = 2^(u_i - u_e) 2^(u_e - u_j) with
                        // a row factor in [1, 2^60] and column weights in [2^-60, 1] dt_j (warp-uniform)
                        fact[hh] = su[q * 32] - ue < 60.f;
                        ar[hh] = fast_exp2(uih - ue);
                    } else {  // strictly below: both factors <= 1
                        ar[hh] = fast_exp2(fminf(uih - ue, 0.f));
                    }
                }
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t v[16];
                    tmem_ld16(cb + 32 * q + 16 * hf, v);
                    tmem_ld_wait16(v);
                    uint32_t o[16];  // M_0 (o[0..7]) and M_1 (o[8..15]) of these 16 positions
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float* su = hh ? su1 : su0;
                        const float uih = hh ? ui[1] : ui[0];
                        const float arh = hh ? ar[1] : ar[0];
                        const bool fh = hh ? fact[1] : fact[0];
                        const int jb = q * 32 + 16 * hf;  // first column of this half
                        float m[16];
                        if (!diag || fh) {
                            // the 16 column weights first (four 16-byte loads, all issued before any use)
                            float4 bc[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) bc[i] = *reinterpret_cast<const float4*>(su + 256 + jb + 4 * i);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {  // packed pairs: half the multiply instructions
                                const float2 ar2 = make_float2(arh, arh);
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
                            float4 uj[4], dj[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uj[i] = *reinterpret_cast<const float4*>(su + jb + 4 * i);
                                dj[i] = *reinterpret_cast<const float4*>(su + 128 + jb + 4 * i);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                m[4 * i + 0] = __uint_as_float(v[4 * i + 0]) * fast_exp2(fminf(uih - uj[i].x, 0.f)) * dj[i].x;
                                m[4 * i + 1] = __uint_as_float(v[4 * i + 1]) * fast_exp2(fminf(uih - uj[i].y, 0.f)) * dj[i].y;
                                m[4 * i + 2] = __uint_as_float(v[4 * i + 2]) * fast_exp2(fminf(uih - uj[i].z, 0.f)) * dj[i].z;
                                m[4 * i + 3] = __uint_as_float(v[4 * i + 3]) * fast_exp2(fminf(uih - uj[i].w, 0.f)) * dj[i].w;
                            }
                        }
                        if (diag) {  // causal mask: column jb + jj is kept for rows r >= it
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) m[jj] = (jb + jj <= r) ? m[jj] : 0.f;
                        }
                        // pack, and fold the magnitudes in a tree (short dependency chains)
                        uint32_t pk[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) pk[jj] = pack_f16x2(m[2 * jj], m[2 * jj + 1]);
                        __half2 t0 = __hmax2(__habs2(*reinterpret_cast<__half2*>(&pk[0])), __habs2(*reinterpret_cast<__half2*>(&pk[1])));
                        __half2 t1 = __hmax2(__habs2(*reinterpret_cast<__half2*>(&pk[2])), __habs2(*reinterpret_cast<__half2*>(&pk[3])));
                        __half2 t2 = __hmax2(__habs2(*reinterpret_cast<__half2*>(&pk[4])), __habs2(*reinterpret_cast<__half2*>(&pk[5])));
                        __half2 t3 = __hmax2(__habs2(*reinterpret_cast<__half2*>(&pk[6])), __habs2(*reinterpret_cast<__half2*>(&pk[7])));
                        mx = __hmax2(mx, __hmax2(__hmax2(t0, t1), __hmax2(t2, t3)));
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) o[8 * hh + jj] = pk[jj];
                    }
                    tmem_st16(cb + 32 * q + 16 * hf, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar->m_ready);
            mbar_arrive(&bar->u_free[ub]);
        }
        flag_f16_range(err, hmax_to_float(mx));
    } else if (warp < 16) {
        // ------------------------------------------------------ state warpgroups SX = 0, 1
        // Token role: row t = r of the x tile of head SX.  State role: TMEM lane r = state row
        // (head r / 64, p = r % 64), columns n of half SX.  A failed wait turns the remaining work into
        // no-ops but keeps every arrival.
        const int SX = (warp - 8) >> 2;
        const int r = threadIdx.x - 256 - 128 * SX;
        const int hs = r >> 6;  // head of the state row
        const uint32_t lane_base = (uint32_t)(((warp - 8) & 3) * 32) << 16;
        const int64_t PN = (int64_t)d.headdim * N;
        const float* init = a.init + (((int64_t)b * a.state_spans + (int64_t)s * a.state_step) * HC + hl0 + hs) * PN +
                            (int64_t)(r & 63) * N;
        constexpr int NC = N / 64;  // 32-column chunks of the state row per warpgroup
        bool ok = true;
        __half2 mx = __floats2half2_rn(0.f, 0.f);
        float prev_raw[2] = {0.f, 0.f};  // raw dA_cumsum of the token before this sub-block (same chunk)
        uint4 xr[8];                     // this thread's bf16 x row (head SX) of the current sub-block
        for (int k = 0; k <= nsb; ++k) {
            // (d) of the previous sub-block: once S has read X', the float16 x row for M X
            if (k >= 1) {
                ok = ok && wait_bounded<false>(&bar->s_done, (k - 1) & 1, abort_flag, err, 51, wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    uint8_t* xrow = xtile((k - 1) % K::NX, SX);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&xr[ch]);
                        uint4 o;
                        uint32_t* o4 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(p2[e]);
                            o4[e] = pack_f16x2(f.x, f.y);
                        }
                        hmax_abs4(mx, o.x, o.y, o.z, o.w);
                        *reinterpret_cast<uint4*>(xrow + sw128_offset(r, ch)) = o;
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(&bar->xf_ready);
            }
            if (k == nsb) break;
            const int64_t t0 = ts + (int64_t)k * 128;
            const int nv = (int)min((int64_t)128, te - t0);
            const int xs = k % K::NX;
            const int ub = k % 3;
            // (a) decays: u, dt and the column weight of head SX for token row r; u_last of both heads
            if (k >= 3) ok = ok && wait_bounded<false>(&bar->u_free[ub], ((k / 3) - 1) & 1, abort_flag, err, 52, wait_ns);
            ok = ok && wait_bounded<false>(&bar->x_full[xs], (k / K::NX) & 1, abort_flag, err, 53, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            const int p0 = (int)(t0 % Q);
            const bool valid = r < nv;
            float ulast[2] = {0.f, 0.f};
            float w = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float* scs = reinterpret_cast<const float*>(smem + K::OFF_CD + (2 * xs + hh) * 1024);
                const float prev = (p0 > 0) ? prev_raw[hh] : 0.f;
                if (ok) {
                    ulast[hh] = sub_block_decay(scs, prev, p0, Q, nv - 1);
                    if (hh == SX) {
                        float u = ulast[hh], dtv = 0.f, bcol = 0.f;
                        if (valid) {
                            u = sub_block_decay(scs, prev, p0, Q, r);
                            dtv = scs[128 + r];
                            // column weight of the factorized mask: 2^(u_end - u_r) dt_r, end = last valid
                            // position of r's 32-block
                            const float uend = sub_block_decay(scs, prev, p0, Q, min(r | 31, nv - 1));
                            bcol = fast_exp2(fminf(uend - u, 0.f)) * dtv;
                            w = fast_exp2(fminf(ulast[hh] - u, 0.f)) * dtv;
                        }
                        float* su = sU + (2 * ub + hh) * 512;
                        su[r] = u;
                        su[128 + r] = dtv;
                        su[256 + r] = bcol;
                    }
                    prev_raw[hh] = scs[nv - 1];
                }
            }
            mbar_arrive(&bar->uv_ready[ub]);
            // (b) columns of half SX of the state row r: the float16 copy for Yst = C H^T, and 2^(u_last)
            //     times them in TMEM
            if (k >= 1) {
                ok = ok && wait_bounded<false>(&bar->ys_done, (k - 1) & 1, abort_flag, err, 54, wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
            }
            if (ok) {
                const float dsb = exp2f(hs ? ulast[1] : ulast[0]);  // (a select: no local-memory array)
                uint8_t* hrow = smem + K::OFF_H;
#pragma unroll 1
                for (int c = SX * NC; c < SX * NC + NC; ++c) {
                    uint32_t v[32];
                    if (k == 0) {
                        const float4* src = reinterpret_cast<const float4*>(init + 32 * c);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 f = src[i];
                            v[4 * i] = __float_as_uint(f.x);
                            v[4 * i + 1] = __float_as_uint(f.y);
                            v[4 * i + 2] = __float_as_uint(f.z);
                            v[4 * i + 3] = __float_as_uint(f.w);
                        }
                    } else {
                        tmem_ld32(tm + lane_base + K::T_H + 32 * c, v);
                        tmem_ld_wait(v);
                    }
                    // columns n = 32 c .. 32 c + 31: K-block c / 2, 16-byte chunks 4 (c % 2) .. + 3
                    uint8_t* kb = hrow + (c >> 1) * kTile;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 o;
                        o.x = pack_f16x2(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1]));
                        o.y = pack_f16x2(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3]));
                        o.z = pack_f16x2(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5]));
                        o.w = pack_f16x2(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7]));
                        hmax_abs4(mx, o.x, o.y, o.z, o.w);
                        *reinterpret_cast<uint4*>(kb + sw128_offset(r, 4 * (c & 1) + q4)) = o;
                    }
                    const float2 dsb2 = make_float2(dsb, dsb);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {  // packed pairs
                        const float2 f = fmul2(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), dsb2);
                        v[2 * i] = __float_as_uint(f.x);
                        v[2 * i + 1] = __float_as_uint(f.y);
                    }
                    tmem_st32(tm + lane_base + K::T_H + 32 * c, v);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
            }
            mbar_arrive(&bar->h_ready);
            // (c) X' = w x over the bf16 x row of head SX (kept in registers for (d); read on every path, so
            //     that it is dead between (d) and here)
            uint8_t* xrow = xtile(xs, SX);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) xr[ch] = *reinterpret_cast<const uint4*>(xrow + sw128_offset(r, ch));
            if (ok) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&xr[ch]);
                    uint4 o;
                    uint32_t* o4 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = fmul2(__bfloat1622float2(p2[e]), make_float2(w, w));
                        o4[e] = pack_f16x2(f.x, f.y);
                    }
                    hmax_abs4(mx, o.x, o.y, o.z, o.w);
                    *reinterpret_cast<uint4*>(xrow + sw128_offset(r, ch)) = o;
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&bar->xs_ready);
        }
        flag_f16_range(err, hmax_to_float(mx));
    } else if (warp < 20) {
        // ------------------------------------------------------ epilogue: y = Y + 2^u Yst, both heads
        const int r = threadIdx.x - 512;
        const uint32_t lane_base = (uint32_t)((warp - 16) * 32) << 16;
        bool ok = true;
        for (int k = 0; k < nsb; ++k) {
            const int64_t t0 = ts + (int64_t)k * 128;
            const int nv = (int)min((int64_t)128, te - t0);
            const int ub = k % 3;
            ok = ok && wait_bounded<false>(&bar->y_full, k & 1, abort_flag, err, 61, wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            float e[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) e[hh] = fast_exp2(fminf(sU[(2 * ub + hh) * 512 + r], 0.f));
            mbar_arrive(&bar->u_free[ub]);
            if (ok) {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const int64_t row = (((int64_t)b * d.seqlen + t0 + r) * H + h0 + hh) * 64;
                    uint4* yrow = reinterpret_cast<uint4*>(a.y + row);
                    const float eh = hh ? e[1] : e[0];
#pragma unroll 1
                    for (int qq = 0; qq < 4; ++qq) {  // 16 channels at a time
                        uint32_t yv[16], sv[16];
                        tmem_ld16(tm + lane_base + K::T_Y + 64 * hh + 16 * qq, yv);
                        tmem_ld16(tm + lane_base + K::T_YS + 64 * hh + 16 * qq, sv);
                        tmem_ld_wait16(sv);
                        tmem_ld_wait16(yv);
                        if (hh == 1 && qq == 3) {
                            tc_fence_before();
                            mbar_arrive(&bar->y_free);  // Y and Yst may be overwritten
                        }
                        if (r < nv) {
                            uint4 ov[2];
#pragma unroll
                            for (int ch = 0; ch < 2; ++ch) {
                                uint32_t* o4 = reinterpret_cast<uint32_t*>(&ov[ch]);
#pragma unroll
                                for (int e2 = 0; e2 < 4; ++e2) {
                                    const int i = ch * 8 + 2 * e2;
                                    const float2 f = ffma2(make_float2(eh, eh),
                                                           make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])),
                                                           make_float2(__uint_as_float(yv[i]), __uint_as_float(yv[i + 1])));
                                    o4[e2] = pack_bf16x2(f.x, f.y);
                                }
                            }
                            if (a.y32) {
                                st_global_32B(yrow + 2 * qq, ov[0], ov[1]);
                            } else {
                                yrow[2 * qq] = ov[0];
                                yrow[2 * qq + 1] = ov[1];
                            }
                        }
                    }
                }
            } else {
                mbar_arrive(&bar->y_free);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tm, K::TCOLS);
}

template <int N>
int launch_pair_n(const __nv_bfloat16* x, const __half* B, const __half* C, const PairArgs& a, cudaStream_t s) {
    const Dims& d = a.d;
    CUtensorMap tx, tb, tc;
    const uint64_t dx[4] = {(uint64_t)d.headdim, (uint64_t)d.nheads, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint64_t dbc[4] = {(uint64_t)d.dstate, (uint64_t)d.ngroups, (uint64_t)d.seqlen, (uint64_t)d.batch};
    const uint32_t box_in[4] = {64, 1, 128, 1};
    if (!make_tmap_16b_4d(&tx, x, dx, box_in) || !make_tmap_16b_4d(&tb, B, dbc, box_in) ||
        !make_tmap_16b_4d(&tc, C, dbc, box_in))
        return SSD_ERR_CUDA;
    const int smem = PCfg<N>::SMEM;
    if (ensure_smem_limit(reinterpret_cast<const void*>(chunk_scan_pair_kernel<N>), smem) != SSD_OK) return SSD_ERR_CUDA;
    dim3 grid(d.hcount / 2, a.nspans, d.batch);
    launch_begin(kKindChunkScan, s);
    const cudaError_t le = launch_dependent(chunk_scan_pair_kernel<N>, grid, dim3(kThreads), smem, s, tx, tb, tc, a);
    const int r = launch_end(kKindChunkScan, s);
    return le != cudaSuccess ? SSD_ERR_CUDA : r;
}

}  // namespace

bool chunk_scan_pair_supported(const Dims& d, const OutOpts& oo) {
    return (d.dstate == 64 || d.dstate == 128) && ((d.nheads / d.ngroups) % 2 == 0) && d.head0 % 2 == 0 &&
           d.hcount % 2 == 0 && oo.Dp == nullptr && oo.z == nullptr;
}

int launch_chunk_scan_pair(const __nv_bfloat16* x, const __half* B, const __half* C, const float* dtt,
                           const float* cs, const float* D, const float* span_states, int span_chunks, const Dims& d,
                           __nv_bfloat16* y, const Ctl& ctl, cudaStream_t s, int state_step) {
    PairArgs a;
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
    a.ctl = ctl;
    switch (d.dstate) {
        case 64: return launch_pair_n<64>(x, B, C, a, s);
        case 128: return launch_pair_n<128>(x, B, C, a, s);
        default: return SSD_ERR_UNSUPPORTED;
    }
}

}  // namespace ssd
