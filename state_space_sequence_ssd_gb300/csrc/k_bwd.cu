// k_bwd.cu -- backward pass of the chunked scan on tcgen05 tensor cores: the
// gradients of a scalar loss with respect to x, dt, A, B, C, D and the initial
// state, given dLoss/dy and dLoss/dfinal.
//
// The pages describe no backward pass; they only note that training speed
// depends on one.  This is the reverse mode of the recurrence the forward
// computes, in the forward's chunked shape (disconfirmai.com page "Jane Street
// ML Engineers Map Mamba-2 Recurrent State Computation to Tensor Cores with
// cuTile", three-kernel and jump-formula paragraphs; devotd.net page on the
// Mamba-2 cuTile forward kernels, section 2).  Per (batch, head), over blocks
// of T = 128 tokens, with c the inclusive cumulative log2 decay inside the
// block, c_e its last value, L[r][i] = 2^(c_r - c_i) for r >= i (else 0), h0
// the state before the block and mu the gradient flowing into the state after
// the block from later tokens (h0 and mu come from the forward and the reverse
// hops over blocks):
//
//   G   = (L o C B^T)^T dY + diag(2^(c_e - c)) B mu        row i: lam_i^T B_i
//   dx  = diag(dt) G + D dY
//   Wd  = L o (dY X^T) o dt_j                               (dt on the columns)
//   dC += diag(2^c) dY h0^T + Wd B                          summed over the group's heads
//   dB += diag(dt 2^(c_e - c)) X mu^T + Wd^T C
//   ddt = A dl + s,   s_t = x_t . G_t
//
// where dl_t = exp(dt_t A) <lam_t, state_{t-1}> is the gradient of the step log-decay dt_t A.
// Splitting lam_t and state_{t-1} at the block's ends keeps every sum inside the block:
//   dl_t = 2^(c_e) <mu, h0> + sum_{j<t} v_j + sum_{r>=t} (rho1_r + rho2_r - sigma_r)
//   v_j     = dt_j 2^(c_e - c_j) x_j . (B mu)_j          (mu reaching back to token j)
//   rho2_r  = 2^(c_r) dy_r . (C h0)_r                    (h0 reaching token r: a fourth product C h0)
//   rho1_r  = sum_j Wd[r][j] (C_r . B_j)                 (pairs inside the block, rows of Wd o C B^T)
//   sigma_r = dt_r x_r . ((L o C B^T)^T dY)_r            (the same pairs by columns)
// (a prefix over the whole sequence of the per-token differences would telescope to the same value
// but accumulate the operands' rounding over every earlier token).  dA = sum of dt_t dl_t over
// tokens and batch, dD = sum of x . dy: per (b, h, block) partial sums, added up in a fixed order
// by bwd_reduce_kernel.
//
// One CTA per (block, group slice, batch) walks hpg / S heads of the group, with dB and dC
// accumulated in TMEM across them; the S CTAs of a group form a thread-block cluster and add their
// partial dB and dC through distributed shared memory in rank order, so the result is written once,
// without atomics and in a fixed order (S = 1: no cluster).  Per head the 512 worker threads run
// the conversions (x and dy to float16 tiles, the two scaled tiles 2^c dy and dt 2^(c_e - c) x, h0 and
// mu to float16), the mask (one thread per row and column quarter: M' = L o C B^T and Wd to float16
// tiles) and the epilogue, one after another.  One more warp issues the products, each as soon as the
// phase that writes its operands has signalled (mbarriers both ways): dY X^T once x and dy are in
// float16 (before the scaled rows), the unmasked dC / dB terms during the mask, B mu and C h0 once the
// mask has read C B^T and dY X^T, G after it, then the masked dC / dB terms and the next head's C B^T
// while the workers run the epilogue and the next head's conversions.  Another warp runs the
// dt-gradient scans of each head from the epilogue's per-row partial sums, while the workers go on
// to the next head (they wait for it only before the next mask overwrites those sums).  The next
// head's inputs (raw x and dy rows, its h0 and mu -- already float16, in the tiles' swizzled order --
// its dA_cumsum and dt rows, D and A) are copied with cp.async into tiles the products have finished
// with as soon as they retire, so their loads overlap the epilogue.
// Operands are float16 (the inputs exactly, the derived tiles rounded once), accumulation float32.
#include "common.cuh"
#include "scan_util.cuh"
#include "sm100.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int T = kBwdBlock;     // tokens per block = the products' M
constexpr int kP = 64;           // headdim
constexpr int kWorkers = 512;    // four warpgroups: warp w owns TMEM lanes 32 (w % 4) .. +31, column quarter w / 4
constexpr int kIssuerWarp = kWorkers / 32;  // one more warp: its first thread issues the products
constexpr int kScanWarp = kIssuerWarp + 1;  // and another: the dt-gradient scans of each head
constexpr int kThreads = kWorkers + 64;
constexpr int kNQ = kWorkers / 128;  // column quarters of a row (mask, epilogue) and row parts (conversions)
constexpr int kPanel = T * 128;  // one 64-column float16 panel of a T-row tile (16 KB)
constexpr int kPanelP = kP * 128;  // one 64-column float16 panel of a P-row tile (8 KB)

template <int N>
struct BwdCfg {
    static constexpr int NP = N / 64;                    // 64-column panels of a B / C / state tile
    static constexpr int OFF_C = 0;                      // C  [t][n]
    static constexpr int OFF_B = OFF_C + NP * kPanel;    // B  [t][n]
    static constexpr int OFF_X = OFF_B + NP * kPanel;    // x  [t][p]
    static constexpr int OFF_DY = OFF_X + kPanel;        // dy [t][p]
    static constexpr int OFF_DYS = OFF_DY + kPanel;      // 2^c dy
    static constexpr int OFF_XS = OFF_DYS + kPanel;      // dt 2^(c_e - c) x
    static constexpr int OFF_H0 = OFF_XS + kPanel;       // h0 [p][n]
    static constexpr int OFF_MU = OFF_H0 + NP * kPanelP; // mu [p][n]
    static constexpr int OFF_M = OFF_MU + NP * kPanelP;  // M' [r][i]; the epilogue's reductions after the products
    static constexpr int OFF_W = OFF_M + 2 * kPanel;     // Wd [r][j]
    static constexpr int OFF_CS = OFF_W + 2 * kPanel;    // cs[T], dt[T]
    static constexpr int OFF_BAR = OFF_CS + 2 * T * 4;   // eleven mbarriers, TMEM base, abort flag, warp sums
    static constexpr int SMEM = OFF_BAR + 192 + 1024;    // + slack to align the base to 1024 bytes
    static_assert(SMEM <= 232448, "shared memory budget");
};

// TMEM columns (all 512): C B^T and dY X^T while the mask reads them, then G, B mu and C h0 in
// their place (B mu and C h0 over the columns the mask reads first, G over the rest); the dC and dB
// accumulators over the group's heads
constexpr uint32_t T_CB = 0, T_DX = 128, T_GMU = 0, T_G = 64, T_YS = 128, T_DC = 256, T_DB = 384;

constexpr uint32_t kIdescTT = idesc_fp16(128, 128, false, false);  // C B^T, dY X^T: both K-major
constexpr uint32_t kIdescG = idesc_fp16(128, 64, true, true);      // M'^T dY: both MN-major
constexpr uint32_t kIdescP = idesc_fp16(128, 64, false, false);    // B mu, C h0: both K-major over n

struct BwdArgs {
    const __nv_bfloat16 *x, *dy;
    const __half *B16, *C16;
    const float *cs, *dtt, *D;
    const __half *h0, *mu;  // block-start states and block-end gradients, float16 (b, nblk, H, P, N)
    const float* A;
    __nv_bfloat16* dx;
    float *ddt, *dB, *dC, *dap, *xdy;  // dap, xdy: per (b, h, block) partial sums of dt dl and x . dy
    Dims d;
    Ctl ctl;
    int slices;  // S: CTAs (a cluster) per (block, group), each with hpg / S heads
};

// C B^T (K = n) of the block into its TMEM columns; one thread issues it
template <int N>
__device__ __forceinline__ void issue_cb(uint32_t tm, uint32_t sC, uint32_t sB) {
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
        mma_ss(tm + T_CB, desc_sw128(sC + off, 16, 1024), desc_sw128(sB + off, 16, 1024), kIdescTT, kk > 0);
    }
}

// bfloat16 pair (low, high) -> float2
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// 4-byte asynchronous copy global -> shared (visible to the issuing thread after cp_async_wait_all)
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Barrier of the kWorkers worker threads only (named barrier 1; the issuer warp does not take part).
__device__ __forceinline__ void worker_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWorkers) : "memory"); }

// The same barrier, returning whether `p` holds on every worker thread.
__device__ __forceinline__ bool worker_and(bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, q;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, a;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(kWorkers)
        : "memory");
    return r != 0;
}

// One arrival per warp on `bar` (initialised with one arrival per worker warp), after every lane's
// writes: __syncwarp orders them before the first lane's release.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) bwd_chunk_kernel(BwdArgs a) {
    using K = BwdCfg<N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* scs = reinterpret_cast<float*>(smem + K::OFF_CS);
    float* sdt = scs + T;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + K::OFF_BAR);
    uint64_t* stall_bar = bar;  // never completed: the test hook's wait runs out on it
    // workers -> issuer, one arrival per worker warp and head: the float16 x and dy tiles are written; all
    // float16 input tiles are written; the mask
    // has read C B^T and dY X^T; M' and Wd are written; G, B mu and C h0 are read
    uint64_t *ev_red = bar + 20, *ev_scanned = bar + 21;  // the epilogue's partial sums are in place; scanned
    uint64_t *ev_xd = bar + 19, *ev_in = bar + 1, *ev_tfree = bar + 7, *ev_mask = bar + 2, *ev_epi = bar + 3;
    // issuer -> workers, one commit per head: C B^T and dY X^T; G, B mu and C h0; and, once, every product
    uint64_t *mm1 = bar + 4, *mm2 = bar + 5, *mm_done = bar + 6;
    uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(bar + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 9);
    float* wsum = reinterpret_cast<float*>(bar + 10);  // per-warp partial sums of <mu, h0> (16 floats)
    float* hconst = wsum + 16;                        // the current head's D and A
    // the next head's dA_cumsum and dt rows, D and A, copied during the epilogue into the upper half of the
    // M' tile (free from the products' reading it until the next head's mask)
    float* stg = reinterpret_cast<float*>(smem + K::OFF_M + kPanel);

    const Dims& d = a.d;
    const int S = a.slices;
    const int blk = blockIdx.x, g = blockIdx.y / S, slice = blockIdx.y % S, b = blockIdx.z;
    const int H = d.nheads, G = d.ngroups, hpg = H / G, hps = hpg / S;
    const int64_t L = d.seqlen;
    const int64_t t0 = (int64_t)blk * T;
    const int64_t rowlen = (int64_t)d.nchunks * T;  // cs / dt / s / q row length per (b, h)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qw = warp & 3, qc = warp >> 2;         // TMEM lane quarter, column quarter
    const int r = 32 * qw + lane;                    // this thread's row in the mask and the epilogue
    const uint32_t lane_base = (uint32_t)(32 * qw) << 16;
    int* const err = a.ctl.err;
    const uint64_t wait_ns = a.ctl.wait_ns;

    if (tid == 0) {
        mbar_init(stall_bar, 1);
        mbar_init(ev_xd, kWorkers / 32);
        mbar_init(ev_red, kWorkers / 32);
        mbar_init(ev_scanned, 1);
        mbar_init(ev_in, kWorkers / 32);
        mbar_init(ev_tfree, kWorkers / 32);
        mbar_init(ev_mask, kWorkers / 32);
        mbar_init(ev_epi, kWorkers / 32);
        mbar_init(mm1, 1);
        mbar_init(mm2, 1);
        mbar_init(mm_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_sh, 512);
        tmem_relinquish();
    }
    const uint32_t sC = smem_u32(smem + K::OFF_C), sB = smem_u32(smem + K::OFF_B);
    const uint32_t sX = smem_u32(smem + K::OFF_X), sDY = smem_u32(smem + K::OFF_DY);
    const uint32_t sDYS = smem_u32(smem + K::OFF_DYS), sXS = smem_u32(smem + K::OFF_XS);
    const uint32_t sH0 = smem_u32(smem + K::OFF_H0), sMU = smem_u32(smem + K::OFF_MU);
    const uint32_t sM = smem_u32(smem + K::OFF_M), sW = smem_u32(smem + K::OFF_W);
    constexpr uint32_t kIdescN = idesc_fp16(128, N, false, true);  // dY' h0^T, Wd B, X' mu^T
    constexpr uint32_t kIdescNT = idesc_fp16(128, N, true, true);  // Wd^T C

    // Inputs of head hh: its x and dy rows (bfloat16) into the swizzled positions of the XS / DYS
    // tiles (zeros past the sequence end), h0 and mu (float16 rows p) straight into the H0 / MU tiles,
    // this thread's dA_cumsum (tid < T) or dt value (T <= tid < 2 T) of the block and (thread 0) the head's
    // D and A into `stg`: copies in flight while the current head finishes, none held in registers.
    const uint32_t stg_s = smem_u32(stg);
    auto prefetch = [&](int hh) {
        const int64_t crow = ((int64_t)b * H + hh) * rowlen + t0;
        if (tid < 2 * T) cp_async4(stg_s + 4 * tid, tid < T ? a.cs + crow + tid : a.dtt + crow + tid - T);
        if (tid == 0) {
            if (a.D != nullptr) cp_async4(stg_s + 8 * T, a.D + hh);
            else stg[2 * T] = 0.f;
            cp_async4(stg_s + 8 * T + 4, a.A + hh);
        }
#pragma unroll
        for (int i = 0; i < T * 8 / kWorkers; ++i) {
            const int c = tid + i * kWorkers;
            const int row = c >> 3, ch = c & 7;
            const int64_t tok = t0 + row;
            const int64_t o = ((b * L + (tok < L ? tok : 0)) * H + hh) * (int64_t)kP + ch * 8;
            const uint32_t nb = tok < L ? 16u : 0u;
            cp_async16(sXS + sw128_offset(row, ch), a.x + o, nb);
            cp_async16(sDYS + sw128_offset(row, ch), a.dy + o, nb);
        }
        const int64_t srow = (((int64_t)b * d.nchunks + blk) * H + hh) * (int64_t)kP * N;
#pragma unroll
        for (int i = 0; i < kP * N / 8 / kWorkers; ++i) {  // 16-byte chunks: 8 columns n of row p
            const int c = tid + i * kWorkers;
            const int p = c / (N / 8), cc = c % (N / 8);
            const uint32_t so = (cc >> 3) * kPanelP + sw128_offset(p, cc & 7);
            cp_async16(sH0 + so, a.h0 + srow + (int64_t)c * 8, 16u);
            cp_async16(sMU + so, a.mu + srow + (int64_t)c * 8, 16u);
        }
        cp_async_commit();
    };
    // the block's B and C rows (float16 copies), once for all heads of the group, and the first head's
    // inputs: all copies in flight together
    for (int c = tid; c < T * N / 8; c += kThreads) {
        const int row = c / (N / 8), cc = c % (N / 8);
        const int64_t tok = t0 + row;
        const int64_t o = ((b * L + (tok < L ? tok : 0)) * G + g) * (int64_t)N + cc * 8;
        const uint32_t nb = tok < L ? 16u : 0u;  // zeros past the sequence end
        const uint32_t so = (cc >> 3) * kPanel + sw128_offset(row, cc & 7);
        cp_async16(sB + so, a.B16 + o, nb);
        cp_async16(sC + so, a.C16 + o, nb);
    }
    cp_async_commit();
    if (warp < kIssuerWarp) {
        prefetch(g * hpg + slice * hps);
        asm volatile("cp.async.wait_group 1;" ::: "memory");  // B and C landed; the head's inputs may not have
    } else {
        cp_async_wait_all();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_sh;
    bool ok = true;
    if (a.ctl.stall && tid == 0) ok = mbar_wait_bounded(stall_bar, 0, abort_flag, err, 60, wait_ns);
    ok = __syncthreads_and(ok);


    __half2 mx = __floats2half2_rn(0.f, 0.f);  // largest |value| converted to float16 (range flag)
    bool fin = true;                           // the issuer's final drain

    if (warp == kIssuerWarp) {
        // ---- the products, issued by one thread in the order the workers' phases need them; each waits only
        //      for the phase that writes its operands, so the tensor pipe works while the workers convert,
        //      mask and run the epilogue
        if (lane == 0) {
#pragma unroll 1
            for (int k = 0; k < hps && ok; ++k) {
                const uint32_t par = k & 1;
                // this head's float16 x and dy tiles are written
                if (!(ok = mbar_wait_bounded(ev_xd, par, abort_flag, err, 68, wait_ns))) break;
                tc_fence_after();
                if (k == 0) issue_cb<N>(tm, sC, sB);  // later heads': issued after the previous epilogue's reads
#pragma unroll
                for (int kk = 0; kk < kP / 16; ++kk)  // dY X^T (K = p)
                    mma_ss(tm + T_DX, desc_sw128(sDY + kk * 32, 16, 1024), desc_sw128(sX + kk * 32, 16, 1024),
                           kIdescTT, kk > 0);
                mma_commit(mm1);
                // the scaled x and dy, h0 and mu are in place too
                if (!(ok = mbar_wait_bounded(ev_in, par, abort_flag, err, 64, wait_ns))) break;
                tc_fence_after();
                // the dC / dB terms that need no mask, dY' h0^T and X' mu^T (K = p): they run during the mask
#pragma unroll
                for (int kk = 0; kk < kP / 16; ++kk) {
                    mma_ss(tm + T_DC, desc_sw128(sDYS + kk * 32, 16, 1024), desc_sw128(sH0 + kk * 2048, kPanelP, 1024),
                           kIdescN, k > 0 || kk > 0);
                    mma_ss(tm + T_DB, desc_sw128(sXS + kk * 32, 16, 1024), desc_sw128(sMU + kk * 2048, kPanelP, 1024),
                           kIdescN, k > 0 || kk > 0);
                }
                // the mask has read C B^T and dY X^T (it is still writing M' and Wd): B mu and C h0, the
                // epilogue's operands that need no mask, go into their columns
                if (!(ok = mbar_wait_bounded(ev_tfree, par, abort_flag, err, 67, wait_ns))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < N / 16; ++kk) {  // K = n
                    const uint32_t offT = (kk >> 2) * kPanel + (kk & 3) * 32;
                    const uint32_t offP = (kk >> 2) * kPanelP + (kk & 3) * 32;
                    mma_ss(tm + T_GMU, desc_sw128(sB + offT, 16, 1024), desc_sw128(sMU + offP, 16, 1024), kIdescP,
                           kk > 0);
                    mma_ss(tm + T_YS, desc_sw128(sC + offT, 16, 1024), desc_sw128(sH0 + offP, 16, 1024), kIdescP,
                           kk > 0);
                }
                // M' and Wd are written: G = M'^T dY
                if (!(ok = mbar_wait_bounded(ev_mask, par, abort_flag, err, 65, wait_ns))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < T / 16; ++kk)  // K = r
                    mma_ss(tm + T_G, desc_sw128(sM + kk * 2048, kPanel, 1024), desc_sw128(sDY + kk * 2048, kPanel, 1024),
                           kIdescG, kk > 0);
                mma_commit(mm2);
                // dC += Wd B, dB += Wd^T C (K = tokens): they read only the Wd, B and C tiles, which neither the
                // epilogue nor the next head's copies and conversions write; the next head's mask writes Wd only
                // after mm1 of the next head, whose commit covers them
#pragma unroll
                for (int kk = 0; kk < T / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
                    mma_ss(tm + T_DC, desc_sw128(sW + off, 16, 1024), desc_sw128(sB + kk * 2048, kPanel, 1024), kIdescN,
                           1);
                    mma_ss(tm + T_DB, desc_sw128(sW + kk * 2048, kPanel, 1024), desc_sw128(sC + kk * 2048, kPanel, 1024),
                           kIdescNT, 1);
                }
                if (k + 1 < hps) {
                    // the epilogue has read G, B mu and C h0: the next head's C B^T (only the block's B / C) goes
                    // into their columns
                    if (!(ok = mbar_wait_bounded(ev_epi, par, abort_flag, err, 66, wait_ns))) break;
                    tc_fence_after();
                    issue_cb<N>(tm, sC, sB);
                }
            }
            // everything issued retires before TMEM is read or released, whatever happened above
            mma_commit(mm_done);
            fin = mbar_wait_drain(mm_done, 0, err, 63, kDrainNs);
        }
        __syncwarp();
    } else if (warp == kScanWarp) {
        // ---- per head, the dt-gradient scans over the block's tokens (lane l: tokens 4 l .. 4 l + 3), from
        // the partial sums the workers' epilogue leaves in the M' tile: quantity q of token t, quarter qc at
        // red[(q kNQ + qc) T + t] (x . G, x . B mu, dy . C h0, the rho1 pairs, x . dy), then c_e, 2^(c_e),
        // <mu, h0> and A.  dl_t = 2^(c_e) <mu, h0> + (v before t) + (w from t on).
        const float* red = reinterpret_cast<const float*>(smem + K::OFF_M);
#pragma unroll 1
        for (int k = 0; k < hps && ok; ++k) {
            const int h = g * hpg + slice * hps + k;
            if (!(ok = mbar_wait_bounded(ev_red, k & 1, abort_flag, err, 69, wait_ns))) break;
            const float* tail = red + 5 * kNQ * T;
            const float ce = tail[0], ece = tail[1], hmu_all = tail[2], Ah = tail[3];
            const int64_t crow = ((int64_t)b * H + h) * rowlen + t0;
            auto qsum = [&](int q, int t) {  // over the quarters, in a fixed order
                const float* rq = red + q * kNQ * T + t;
                return (rq[0] + rq[T]) + (rq[2 * T] + rq[3 * T]);
            };
            float sfull[4], v[4], w[4], dtl[4], epv[4], epw[4];
            float pv = 0.f, pw = 0.f, xd = 0.f;  // this lane's running sums
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = 4 * lane + j;
                const float cst = __ldg(a.cs + crow + t), dtt = __ldg(a.dtt + crow + t);
                const float ex = fast_exp2(ce - cst);
                const float sgt = qsum(0, t), smt = qsum(1, t);
                sfull[j] = fmaf(ex, smt, sgt);                                     // x_t . G_t
                v[j] = dtt * ex * smt;                                             // mu's part, at token t
                w[j] = fmaf(fast_exp2(cst), qsum(2, t), qsum(3, t)) - dtt * sgt;  // rho2 + rho1 - sigma
                dtl[j] = dtt;
                xd += qsum(4, t);
                epv[j] = pv;
                epw[j] = pw;
                pv += v[j];
                pw += w[j];
            }
            float iv = pv, iw = pw;  // inclusive scans of the lanes' totals
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float ov = __shfl_up_sync(0xffffffffu, iv, off);
                const float ow = __shfl_up_sync(0xffffffffu, iw, off);
                if (lane >= off) {
                    iv += ov;
                    iw += ow;
                }
            }
            const float bv = iv - pv, bw = iw - pw;           // the lanes before this one
            const float tw = __shfl_sync(0xffffffffu, iw, 31);  // all of w
            float da = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = 4 * lane + j;
                const float dl = fmaf(ece, hmu_all, (bv + epv[j]) + (tw - (bw + epw[j])));
                if (t0 + t < L) a.ddt[((b * L + t0 + t) * H + h)] = fmaf(Ah, dl, sfull[j]);
                da = fmaf(dtl[j], dl, da);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                da += __shfl_xor_sync(0xffffffffu, da, off);
                xd += __shfl_xor_sync(0xffffffffu, xd, off);
            }
            __syncwarp();  // every lane's reads of the partial sums are done
            if (lane == 0) {
                const int64_t o = ((int64_t)b * H + h) * d.nchunks + blk;
                a.dap[o] = da;
                a.xdy[o] = xd;
                mbar_arrive(ev_scanned);
            }
        }
    } else {
#pragma unroll 1
        for (int k = 0; k < hps && ok; ++k) {
            const int h = g * hpg + slice * hps + k;
            const uint32_t par = k & 1;
            // ---- this head's raw inputs (copied during the previous head's epilogue) -> float16 tiles
            cp_async_wait_all();
            if (tid < 2 * T) scs[tid] = stg[tid];  // dA_cumsum then dt: `sdt` follows `scs`
            if (tid == 0) {
                hconst[0] = stg[2 * T];
                hconst[1] = stg[2 * T + 1];
            }
            worker_sync();
            const float ce = scs[T - 1];
            // x and dy to float16 first, so that dY X^T starts while the scaled rows are written (a second
            // read of the raw rows)
            {
                const int rr = tid & (T - 1), hl = tid >> 7;  // row, quarter of the row's 64 channels
#pragma unroll
                for (int j = 0; j < 8 / kNQ; ++j) {
                    const uint32_t so = sw128_offset(rr, (8 / kNQ) * hl + j);
                    const uint4 xv = *reinterpret_cast<const uint4*>(smem + K::OFF_XS + so);
                    const uint4 yv = *reinterpret_cast<const uint4*>(smem + K::OFF_DYS + so);
                    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv);
                    const uint32_t* yw = reinterpret_cast<const uint32_t*>(&yv);
                    uint32_t ox[4], oy[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 xf = bf2_to_f2(xw[e]), yf = bf2_to_f2(yw[e]);
                        ox[e] = pack_f16x2(xf.x, xf.y);
                        oy[e] = pack_f16x2(yf.x, yf.y);
                    }
                    hmax_abs4(mx, ox[0], ox[1], ox[2], ox[3]);
                    hmax_abs4(mx, oy[0], oy[1], oy[2], oy[3]);
                    *reinterpret_cast<uint4*>(smem + K::OFF_X + so) = make_uint4(ox[0], ox[1], ox[2], ox[3]);
                    *reinterpret_cast<uint4*>(smem + K::OFF_DY + so) = make_uint4(oy[0], oy[1], oy[2], oy[3]);
                }
                fence_proxy_async_smem();
                warp_arrive(ev_xd);
                const float wx = sdt[rr] * fast_exp2(ce - scs[rr]);
                const float wy = fast_exp2(scs[rr]);
#pragma unroll
                for (int j = 0; j < 8 / kNQ; ++j) {
                    const uint32_t so = sw128_offset(rr, (8 / kNQ) * hl + j);
                    const uint4 xv = *reinterpret_cast<const uint4*>(smem + K::OFF_XS + so);
                    const uint4 yv = *reinterpret_cast<const uint4*>(smem + K::OFF_DYS + so);
                    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv);
                    const uint32_t* yw = reinterpret_cast<const uint32_t*>(&yv);
                    uint32_t oxs[4], oys[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 xs = fmul2(bf2_to_f2(xw[e]), make_float2(wx, wx));
                        oxs[e] = pack_f16x2(xs.x, xs.y);
                        const float2 ys = fmul2(bf2_to_f2(yw[e]), make_float2(wy, wy));
                        oys[e] = pack_f16x2(ys.x, ys.y);
                    }
                    hmax_abs4(mx, oxs[0], oxs[1], oxs[2], oxs[3]);
                    hmax_abs4(mx, oys[0], oys[1], oys[2], oys[3]);
                    *reinterpret_cast<uint4*>(smem + K::OFF_XS + so) = make_uint4(oxs[0], oxs[1], oxs[2], oxs[3]);
                    *reinterpret_cast<uint4*>(smem + K::OFF_DYS + so) = make_uint4(oys[0], oys[1], oys[2], oys[3]);
                }
            }
            float hmu = 0.f;  // this thread's part of <mu, h0> (over the float16 tiles)
#pragma unroll 1
            for (int i = 0; i < kP * N / 8 / kWorkers; ++i) {
                const int c = tid + i * kWorkers;
                const int p = c / (N / 8), cc = c % (N / 8);
                const uint32_t so = (cc >> 3) * kPanelP + sw128_offset(p, cc & 7);
                const uint4 hq = *reinterpret_cast<const uint4*>(smem + K::OFF_H0 + so);
                const uint4 mq = *reinterpret_cast<const uint4*>(smem + K::OFF_MU + so);
                const __half2* hh2 = reinterpret_cast<const __half2*>(&hq);
                const __half2* mh2 = reinterpret_cast<const __half2*>(&mq);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 hf2 = __half22float2(hh2[e]), mf2 = __half22float2(mh2[e]);
                    hmu = fmaf(hf2.x, mf2.x, fmaf(hf2.y, mf2.y, hmu));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) hmu += __shfl_xor_sync(0xffffffffu, hmu, off);
            if (lane == 0) wsum[warp] = hmu;
            fence_proxy_async_smem();  // the tiles written here (and the copies landed) are read by the products
            warp_arrive(ev_in);
            // ---- C B^T and dY X^T; and the previous head's scans have read the partial sums in the M' tile
            ok = mbar_wait_bounded(mm1, par, abort_flag, err, 61, wait_ns);
            if (k > 0) ok = ok && mbar_wait_bounded(ev_scanned, par ^ 1, abort_flag, err, 70, wait_ns);
            ok = worker_and(ok);
            if (!ok) break;
            tc_fence_after();
            // ---- mask: row r, columns [16 qc, 16 qc + 16) and [64 + 16 qc, 64 + 16 qc + 16) of M' = L o C B^T
            //      and Wd = L o dY X^T o dt_j, the first 64 columns first (all warps' first pieces free the
            //      TMEM columns of B mu and C h0)
            float2 rho1p = make_float2(0.f, 0.f);  // sum_j Wd[r][j] (C_r . B_j) over this quarter: even / odd j
            {
                const float cr = scs[r];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int i0 = 16 * qc + 64 * c2;
                    uint32_t vcb[16], vdx[16];
                    tmem_ld16(tm + lane_base + T_CB + i0, vcb);
                    tmem_ld16(tm + lane_base + T_DX + i0, vdx);
                    tmem_ld_wait16(vcb);
                    tmem_ld_wait16(vdx);
                    if (c2 == 0) {  // this warp's reads of columns 0-63 of C B^T and dY X^T
                        tc_fence_before();
                        warp_arrive(ev_tfree);
                    }
                    uint32_t pm[8], pw[8];
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {  // packed pairs of columns
                        const int i = i0 + jj;
                        const float2 dec = make_float2((i <= r) ? fast_exp2(cr - scs[i]) : 0.f,
                                                       (i + 1 <= r) ? fast_exp2(cr - scs[i + 1]) : 0.f);
                        const float2 cb = make_float2(__uint_as_float(vcb[jj]), __uint_as_float(vcb[jj + 1]));
                        const float2 mv = fmul2(dec, cb);
                        const float2 wv = fmul2(fmul2(dec, make_float2(sdt[i], sdt[i + 1])),
                                                make_float2(__uint_as_float(vdx[jj]), __uint_as_float(vdx[jj + 1])));
                        rho1p = ffma2(wv, cb, rho1p);
                        pm[jj / 2] = pack_f16x2(mv.x, mv.y);
                        pw[jj / 2] = pack_f16x2(wv.x, wv.y);
                    }
#pragma unroll
                    for (int j = 0; j < 2; ++j) {  // columns i0 .. i0 + 15: panel c2, chunks 2 qc + j
                        hmax_abs4(mx, pm[4 * j], pm[4 * j + 1], pm[4 * j + 2], pm[4 * j + 3]);
                        hmax_abs4(mx, pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
                        const uint32_t so = c2 * kPanel + sw128_offset(r, 2 * qc + j);
                        *reinterpret_cast<uint4*>(smem + K::OFF_M + so) =
                            make_uint4(pm[4 * j], pm[4 * j + 1], pm[4 * j + 2], pm[4 * j + 3]);
                        *reinterpret_cast<uint4*>(smem + K::OFF_W + so) =
                            make_uint4(pw[4 * j], pw[4 * j + 1], pw[4 * j + 2], pw[4 * j + 3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            warp_arrive(ev_mask);
            // ---- G, B mu, C h0
            ok = mbar_wait_bounded(mm2, par, abort_flag, err, 62, wait_ns);
            ok = worker_and(ok);
            if (!ok) break;
            tc_fence_after();
            // the committed products have read the XS, DYS, H0 and MU tiles: the next head's inputs go there
            if (k + 1 < hps) prefetch(h + 1);
            // ---- epilogue: row r, channels [16 qc, 16 qc + 16)
            {
                float* red = reinterpret_cast<float*>(smem + K::OFF_M);  // [quantity][quarter][T]; M' is consumed
                const int64_t tok = t0 + r;
                const float ext = fast_exp2(ce - scs[r]), dtr = sdt[r], Dh = hconst[0];
                uint32_t vg[16], vm[16];
                tmem_ld16(tm + lane_base + T_G + 16 * qc, vg);
                tmem_ld16(tm + lane_base + T_GMU + 16 * qc, vm);
                tmem_ld_wait16(vg);
                tmem_ld_wait16(vm);
                // x . G (pairs in the block), x . B mu, x . dy: even / odd channel partial sums
                float2 sg2 = make_float2(0.f, 0.f), sm2 = make_float2(0.f, 0.f), xdy2 = make_float2(0.f, 0.f);
                uint32_t ob[8];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint4 xq = *reinterpret_cast<const uint4*>(smem + K::OFF_X + sw128_offset(r, 2 * qc + j));
                    const uint4 yq = *reinterpret_cast<const uint4*>(smem + K::OFF_DY + sw128_offset(r, 2 * qc + j));
                    const __half2* xh = reinterpret_cast<const __half2*>(&xq);
                    const __half2* yh = reinterpret_cast<const __half2*>(&yq);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {  // packed pairs of channels
                        const int c = 8 * j + 2 * e;
                        const float2 xf = __half22float2(xh[e]), yf = __half22float2(yh[e]);
                        const float2 gi = make_float2(__uint_as_float(vg[c]), __uint_as_float(vg[c + 1]));
                        const float2 gm = make_float2(__uint_as_float(vm[c]), __uint_as_float(vm[c + 1]));
                        sg2 = ffma2(xf, gi, sg2);
                        sm2 = ffma2(xf, gm, sm2);
                        xdy2 = ffma2(xf, yf, xdy2);
                        const float g0 = fmaf(ext, gm.x, gi.x), g1 = fmaf(ext, gm.y, gi.y);
                        ob[4 * j + e] = pack_bf16x2(fmaf(dtr, g0, Dh * yf.x), fmaf(dtr, g1, Dh * yf.y));
                    }
                }
                if (tok < L) {
                    uint4* dst = reinterpret_cast<uint4*>(a.dx + ((b * L + tok) * H + h) * (int64_t)kP + 16 * qc);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        dst[j] = make_uint4(ob[4 * j], ob[4 * j + 1], ob[4 * j + 2], ob[4 * j + 3]);
                }
                uint32_t vy[16];
                tmem_ld16(tm + lane_base + T_YS + 16 * qc, vy);
                tmem_ld_wait16(vy);
                // every TMEM read of this head is done: the next head's C B^T may overwrite these columns
                if (k + 1 < hps) {
                    tc_fence_before();
                    warp_arrive(ev_epi);
                }
                float2 rho22 = make_float2(0.f, 0.f);  // dy_r . (C_r h0) over this quarter: even / odd channels
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint4 yq = *reinterpret_cast<const uint4*>(smem + K::OFF_DY + sw128_offset(r, 2 * qc + j));
                    const __half2* yh = reinterpret_cast<const __half2*>(&yq);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 8 * j + 2 * e;
                        rho22 = ffma2(__half22float2(yh[e]),
                                      make_float2(__uint_as_float(vy[c]), __uint_as_float(vy[c + 1])), rho22);
                    }
                }
                red[(0 * kNQ + qc) * T + r] = sg2.x + sg2.y;
                red[(1 * kNQ + qc) * T + r] = sm2.x + sm2.y;
                red[(2 * kNQ + qc) * T + r] = rho22.x + rho22.y;
                red[(3 * kNQ + qc) * T + r] = rho1p.x + rho1p.y;
                red[(4 * kNQ + qc) * T + r] = xdy2.x + xdy2.y;
                if (tid == 0) {  // what the scans need besides the partial sums
                    float hmu_all = 0.f;
#pragma unroll
                    for (int w4 = 0; w4 < kWorkers / 32; w4 += 4)
                        hmu_all += (wsum[w4] + wsum[w4 + 1]) + (wsum[w4 + 2] + wsum[w4 + 3]);
                    float* tail = red + 5 * kNQ * T;
                    tail[0] = ce;
                    tail[1] = fast_exp2(ce);
                    tail[2] = hmu_all;
                    tail[3] = hconst[1];
                }
                warp_arrive(ev_red);  // the scan warp takes it from here; the workers go on to the next head
                // once every worker is past its reads of this head's dA_cumsum, dt, D and A (the next head's
                // first step writes them)
                worker_sync();
            }
        }
        cp_async_wait_all();  // no copy is still landing when the shared memory is reused or released
    }
    flag_f16_range(err, hmax_to_float(mx));
    // the issuer's drain has seen every product retire (or given up): TMEM may be read, then released
    ok = __syncthreads_and(ok && fin);
    tc_fence_after();
    const int64_t tok = t0 + r;
    if (S == 1) {
        if (ok && warp < kIssuerWarp) {
            // dC and dB rows of this block, summed over the group's heads
#pragma unroll 1
            for (int c = 0; c < N / 64; ++c) {  // this warp's quarter of the columns, 16 at a time
                const int n0 = qc * (N / 4) + 16 * c;
                uint32_t vc[16], vb[16];
                tmem_ld16(tm + lane_base + T_DC + n0, vc);
                tmem_ld16(tm + lane_base + T_DB + n0, vb);
                tmem_ld_wait16(vc);
                tmem_ld_wait16(vb);
                if (tok < L) {
                    float4* dc = reinterpret_cast<float4*>(a.dC + ((b * L + tok) * G + g) * (int64_t)N + n0);
                    float4* db = reinterpret_cast<float4*>(a.dB + ((b * L + tok) * G + g) * (int64_t)N + n0);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        dc[j] = make_float4(__uint_as_float(vc[4 * j]), __uint_as_float(vc[4 * j + 1]),
                                            __uint_as_float(vc[4 * j + 2]), __uint_as_float(vc[4 * j + 3]));
                        db[j] = make_float4(__uint_as_float(vb[4 * j]), __uint_as_float(vb[4 * j + 1]),
                                            __uint_as_float(vb[4 * j + 2]), __uint_as_float(vb[4 * j + 3]));
                    }
                }
            }
        }
    } else {
        // this CTA's partial dC and dB -> shared memory (the tiles are consumed), float32 [2][T][NS]
        constexpr int NS = N + 4;  // padded rows: the float4 stores of a warp fall on different banks
        float* acc = reinterpret_cast<float*>(smem);
        if (ok && warp < kIssuerWarp) {
#pragma unroll 1
            for (int c = 0; c < N / 64; ++c) {  // this warp's quarter of the columns, 16 at a time
                const int n0 = qc * (N / 4) + 16 * c;
                uint32_t vc[16], vb[16];
                tmem_ld16(tm + lane_base + T_DC + n0, vc);
                tmem_ld16(tm + lane_base + T_DB + n0, vb);
                tmem_ld_wait16(vc);
                tmem_ld_wait16(vb);
                float4* sc = reinterpret_cast<float4*>(acc + (int64_t)r * NS + n0);
                float4* sb = reinterpret_cast<float4*>(acc + (int64_t)(T + r) * NS + n0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sc[j] = make_float4(__uint_as_float(vc[4 * j]), __uint_as_float(vc[4 * j + 1]),
                                        __uint_as_float(vc[4 * j + 2]), __uint_as_float(vc[4 * j + 3]));
                    sb[j] = make_float4(__uint_as_float(vb[4 * j]), __uint_as_float(vb[4 * j + 1]),
                                        __uint_as_float(vb[4 * j + 2]), __uint_as_float(vb[4 * j + 3]));
                }
            }
        }
        tc_fence_before();
        cluster_sync();  // every CTA's partial sums are in its shared memory
        // this CTA adds rows [slice T / S, (slice + 1) T / S) of both over the cluster, in rank order
        const int rows = T / S, row0 = slice * rows;
        const uint32_t acc_s = smem_u32(acc);
        for (int it = tid; it < 2 * rows * (N / 4); it += kThreads) {
            const int which = it / (rows * (N / 4)), rem = it % (rows * (N / 4));
            const int row = row0 + rem / (N / 4), c4 = rem % (N / 4);
            const uint32_t off = (uint32_t)(((which * T + row) * NS + 4 * c4) * 4);
            float4 sum = ld_shared_cluster_f4(map_shared_rank(acc_s + off, 0));
            for (int k2 = 1; k2 < S; ++k2) {
                const float4 v = ld_shared_cluster_f4(map_shared_rank(acc_s + off, (uint32_t)k2));
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const int64_t trow = t0 + row;
            if (ok && trow < L) {
                float* dst = (which == 0 ? a.dC : a.dB) + ((b * L + trow) * G + g) * (int64_t)N + 4 * c4;
                *reinterpret_cast<float4*>(dst) = sum;
            }
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ---- dA and dD: one CTA per head adds the per-(batch, block) partial sums in a fixed order

constexpr int kRedThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = (lane < kRedThreads / 32) ? sh[lane] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) sh[32] = v;
    }
    __syncthreads();
    return sh[32];
}

__global__ void __launch_bounds__(kRedThreads) bwd_reduce_kernel(const float* __restrict__ dap,
                                                                 const float* __restrict__ xdy, Dims d,
                                                                 float* __restrict__ dA, float* __restrict__ dD) {
    __shared__ float sh[33];
    const int h = blockIdx.x, tid = threadIdx.x;
    float sa = 0.f, sd = 0.f;
    for (int b = 0; b < d.batch; ++b) {
        const int64_t row = ((int64_t)b * d.nheads + h) * d.nchunks;
        for (int64_t k = tid; k < d.nchunks; k += kRedThreads) {
            sa += dap[row + k];
            sd += xdy[row + k];
        }
    }
    sa = block_sum(sa, sh);
    sd = block_sum(sd, sh);
    if (tid == 0) {
        dA[h] = sa;
        if (dD != nullptr) dD[h] = sd;
    }
}

template <int N>
int launch_bwd_n(const BwdArgs& a0, cudaStream_t s) {
    using K = BwdCfg<N>;
    if (ensure_smem_limit(reinterpret_cast<const void*>(bwd_chunk_kernel<N>), K::SMEM) != SSD_OK) return SSD_ERR_CUDA;
    BwdArgs a = a0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = K::SMEM;
    cfg.stream = s;
    attr.id = cudaLaunchAttributeClusterDimension;
    for (;;) {
        cfg.gridDim = dim3(a.d.nchunks, a.d.ngroups * a.slices, a.d.batch);
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = a.slices;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = a.slices > 1 ? 1 : 0;
        if (a.slices == 1) break;
        // a cluster of S CTAs at this shared-memory size must fit the device; else fewer slices
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, reinterpret_cast<const void*>(bwd_chunk_kernel<N>), &cfg) ==
                cudaSuccess &&
            nclusters > 0)
            break;
        cudaGetLastError();
        a.slices /= 2;
    }
    launch_begin(kKindBwdChunk, s);
    const cudaError_t le = cudaLaunchKernelEx(&cfg, bwd_chunk_kernel<N>, a);
    const int r = launch_end(kKindBwdChunk, s);
    return le != cudaSuccess ? SSD_ERR_CUDA : r;
}

}  // namespace

bool bwd_supported(const Dims& d) {
    return d.headdim == kP && (d.dstate == 64 || d.dstate == 128) && d.chunk_size == T && d.head0 == 0 &&
           d.hcount == d.nheads;
}

int launch_bwd_chunk(const __nv_bfloat16* x, const __nv_bfloat16* dy, const __half* B16, const __half* C16,
                     const float* cs, const float* dtt, const float* A, const float* D, const __half* h0, const __half* mu,
                     const Dims& d, __nv_bfloat16* dx, float* ddt, float* dB, float* dC, float* dap, float* xdy,
                     const Ctl& ctl, cudaStream_t s, int slices) {
    const int hpg = d.nheads / d.ngroups;
    if (!bwd_supported(d) || d.nchunks > 2147483647 || (int64_t)d.ngroups * slices > 65535 || d.batch > 65535 ||
        !(slices == 1 || slices == 2 || slices == 4) || hpg % slices != 0)
        return SSD_ERR_UNSUPPORTED;
    BwdArgs a;
    a.x = x;
    a.dy = dy;
    a.B16 = B16;
    a.C16 = C16;
    a.cs = cs;
    a.dtt = dtt;
    a.D = D;
    a.h0 = h0;
    a.mu = mu;
    a.A = A;
    a.dx = dx;
    a.ddt = ddt;
    a.dB = dB;
    a.dC = dC;
    a.dap = dap;
    a.xdy = xdy;
    a.d = d;
    a.ctl = ctl;
    a.slices = slices;
    return d.dstate == 64 ? launch_bwd_n<64>(a, s) : launch_bwd_n<128>(a, s);
}

int launch_bwd_reduce(const float* dap, const float* xdy, const Dims& d, float* dA, float* dD, cudaStream_t s) {
    launch_begin(kKindBwdReduce, s);
    bwd_reduce_kernel<<<d.nheads, kRedThreads, 0, s>>>(dap, xdy, d, dA, dD);
    return launch_end(kKindBwdReduce, s);
}

}  // namespace ssd
