/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 SSD chunked forward pass.
 *
 * Per head h (group g = h / (nheads / ngroups)) and token t the library
 * computes the selective state-space recurrence
 *
 *     hs_t = exp(dt_t * A_h) * hs_{t-1} + B_t (dt_t * x_t)^T      (N x P state)
 *     y_t  = C_t . hs_t + D_h * x_t
 *
 * in chunks of Q = chunk_size tokens, as three stages:
 *   chunk_cumsum   -- in-chunk cumulative sum of dt*A in log2 units;
 *   fwd_pass_state -- per-chunk states B^T (decay * dt * X) (ssd_chunk_state)
 *                     then the sequential jump across chunks (ssd_state_passing);
 *   compute_out    -- carried-state term, causally masked decayed C B^T X term
 *                     and D skip, fused (ssd_chunk_scan).
 * Sources (web pages, by title and section):
 *   "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to
 *   Tensor Cores with cuTile" (disconfirmai.com) -- three-kernel paragraph and
 *   jump-formula paragraph; devotd.net page on the Mamba-2 cuTile forward
 *   kernels, section 2 (the three kernels and the chunk_cumsum listing) and
 *   section 3 (transposed dA_cumsum / dt layout for contiguous reads).
 *
 * Conventions for every entry point
 * ---------------------------------
 *  * All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees or retains them.  Layouts are dense row-major:
 *        x, y        (batch, seqlen, nheads, headdim)      bfloat16
 *        dt          (batch, seqlen, nheads)               float32, dt > 0
 *        A, D        (nheads,)                             float32
 *        B, C        (batch, seqlen, ngroups, dstate)      bfloat16
 *        dA_cumsum   (batch, nheads, nchunks, chunk_size)  float32, log2 units
 *        dt_t        (batch, nheads, nchunks, chunk_size)  float32
 *        chunk_states, states (batch, nchunks, nheads, headdim, dstate) float32
 *        init_state, final_state (batch, nheads, headdim, dstate)        float32
 *    A state is stored as state[p][n] = hs[n][p] (headdim-major, dstate
 *    contiguous).  nchunks = ceil(seqlen / chunk_size); positions past the
 *    end of the sequence behave as dt = 0 (zero padding).
 *  * bfloat16 tensors are passed as void pointers; each element is an IEEE
 *    bfloat16 (the upper 16 bits of a float32).
 *  * Every call is asynchronous on `stream` (0 = legacy default stream) and
 *    never synchronizes the host.  The return value reports argument
 *    validation and launch errors only; a failed validation launches nothing
 *    and leaves every output untouched.  Device-side errors surface at the
 *    caller's next synchronization; a bounded device wait that gave up is
 *    reported by ssd_get_device_error().
 *  * Value domain: A <= 0 (decay rates) and dt >= 0, so every in-chunk decay
 *    factor 2^(dA_cumsum[i] - dA_cumsum[j]), j <= i, is at most 1; the
 *    kernels exponentiate only such differences and never overflow.  Other
 *    values of A or dt are outside the supported domain.
 *  * Supported shapes: headdim == 64; dstate in {64, 128, 256, 512};
 *    chunk_size in {64, 128, 256}; nheads % ngroups == 0; x, B, C, y and the
 *    float32 tensors 16-byte aligned.  Other shapes return
 *    SSD_ERR_UNSUPPORTED (valid but not implemented) or SSD_ERR_INVALID_ARG.
 *  * Precision: the tensor-core products run on float16 operands with float32
 *    accumulation.  B and C are copied to float16 (exact for magnitudes in
 *    [2^-14, 65504]; larger magnitudes saturate), x is converted the same way
 *    on chip, and the derived operands (decayed masked C B^T, carried state,
 *    decay-scaled x) are rounded once to float16.  Every such conversion is
 *    checked on chip: if any converted value (an input element, or a derived
 *    one: an entry of the masked matrix, of the carried state or of a
 *    decay-scaled x row) exceeds float16's largest finite magnitude 65504,
 *    the library's range flag is raised and ssd_get_device_error() reports
 *    SSD_ERR_RANGE; the outputs of that call are then not reliable.  A
 *    result is never wrong without one of these two reports.  Inputs of
 *    magnitude ~1 with a few thousand tokens stay far inside the range;
 *    inputs scaled by ~256 (or a state that grows without decay to ~65504)
 *    leave it.
 *  * No C++ exception crosses this boundary.  The library keeps no state
 *    between calls other than the optional profiling counters below; calls
 *    on different streams may run concurrently, except ssd_forward_noalloc,
 *    whose calls on one device share one scratch array (see there).
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* null required pointer, non-positive size, misalignment, bad grouping */
    SSD_ERR_UNSUPPORTED = 2, /* well-formed shape outside the implemented set */
    SSD_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    SSD_ERR_NO_MEMORY = 4,   /* workspace allocation failed (ssd_forward) */
    SSD_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see ssd_get_device_error) */
    SSD_ERR_SCRATCH_TOO_SMALL = 6, /* ssd_forward_noalloc: workload larger than its fixed scratch */
    SSD_ERR_RANGE = 7        /* a float16 tensor-core operand left float16's range (see ssd_get_device_error) */
} ssd_status;

/* Size in bytes of the fixed device scratch array used by ssd_forward_noalloc. */
#define SSD_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Static, never-NULL description of a status code. */
SSD_API const char* ssd_status_string(int status);

/*
 * ssd_chunk_cumsum -- the chunk_cumsum stage (devotd.net page, section 2 and
 * its listing: dt tile times A, cumulative sum along the chunk, times log2 e;
 * section 3: the result and dt stored chunk-contiguous).
 *   dA_cumsum[b,h,c,i] = log2(e) * sum_{j<=i} dt[b, c*Q+j, h] * A[h]
 *   dt_t[b,h,c,i]      = dt[b, c*Q+i, h]          (0 past the sequence end)
 * dt: (batch, seqlen, nheads); A: (nheads); outputs (batch, nheads, nchunks, Q).
 */
SSD_API int ssd_chunk_cumsum(const float* dt, const float* A, int batch, int seqlen, int nheads,
                     int chunk_size, float* dA_cumsum, float* dt_t, cudaStream_t stream);

/*
 * ssd_chunk_state -- first half of fwd_pass_state: every chunk's own state
 * contribution (the jump formula h(t+T) = h(t) + B X^T with X's rows
 * pre-scaled by the decay to the chunk end and by dt; disconfirmai.com page,
 * jump-formula paragraph):
 *   chunk_states[b,c,h][p][n] = sum_{i in chunk c} B[b,t_i,g,n] * w_i * x[b,t_i,h,p],
 *   w_i = 2^(dA_cumsum[b,h,c,Q-1] - dA_cumsum[b,h,c,i]) * dt_t[b,h,c,i].
 * dt_t and dA_cumsum are ssd_chunk_cumsum's outputs.  Allocates a
 * stream-ordered float16 copy of B from the library's memory pool (freed on
 * `stream`); returns SSD_ERR_NO_MEMORY if that fails.
 */
SSD_API int ssd_chunk_state(const void* x, const void* B, const float* dt_t, const float* dA_cumsum,
                    int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                    int chunk_size, float* chunk_states, cudaStream_t stream);

/*
 * ssd_state_passing -- second half of fwd_pass_state: the sequential jump
 * across chunks, parallel over the independent (p, n) state entries
 * (devotd.net page, section 2: chunk order kept, independent parts of the
 * state processed in parallel):
 *   h_0 = init_state (zeros if NULL);  states[c] = h_c;
 *   h_{c+1} = 2^(dA_cumsum[b,h,c,Q-1]) * h_c + chunk_states[c];
 *   final_state = h_nchunks (not written if NULL).
 * `states` may alias `chunk_states` (in-place update is supported).
 */
SSD_API int ssd_state_passing(const float* chunk_states, const float* dA_cumsum, const float* init_state,
                      int batch, int nchunks, int nheads, int headdim, int dstate, int chunk_size,
                      float* states, float* final_state, cudaStream_t stream);

/*
 * ssd_chunk_scan -- compute_out: output of every chunk from its chunk-start
 * state, fused so that the Q x Q interaction matrix never leaves the chip
 * (disconfirmai.com page, three-kernel paragraph; devotd.net page, section 2):
 *   y[t_i] = 2^(cs_i) * (C_i . h_c)
 *          + sum_{j<=i} (C_i . B_j) * 2^(cs_i - cs_j) * dt_j * x_j
 *          + D[h] * x_i,          cs = dA_cumsum[b,h,c,:],  h_c = states[b,c,h]
 * D may be NULL (no skip term).  y: (batch, seqlen, nheads, headdim) bfloat16.
 * Allocates stream-ordered float16 copies of B and C from the library's
 * memory pool (freed on `stream`); returns SSD_ERR_NO_MEMORY if that fails.
 */
SSD_API int ssd_chunk_scan(const void* x, const void* B, const void* C, const float* dt_t,
                   const float* dA_cumsum, const float* D, const float* states, int batch,
                   int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk_size,
                   void* y, cudaStream_t stream);

/*
 * ssd_forward -- the whole chunked forward pass: y and the final state from
 * the raw inputs.  D, init_state and final_state may be NULL.  Allocates its
 * workspace stream-ordered on `stream` from a library-owned memory pool per
 * device that keeps freed memory cached for the next call
 * (cudaMallocFromPoolAsync / cudaFreeAsync), and returns SSD_ERR_NO_MEMORY if
 * that fails.  The result equals the recurrence
 * above for any chunk_size; chunk_size only sets the internal tiling.
 */
SSD_API int ssd_forward(const void* x, const float* dt, const float* A, const void* B, const void* C,
                const float* D, const float* init_state, int batch, int seqlen, int nheads,
                int headdim, int ngroups, int dstate, int chunk_size, void* y,
                float* final_state, cudaStream_t stream);

/*
 * ssd_forward_heads -- ssd_forward over the contiguous range of heads
 * [head_begin, head_begin + head_count) of full-size tensors, in place: the
 * multi-GPU split of the pass.  Per batch row, (batch, head) units are
 * independent -- each head reads its own x, dt, A, D and initial state and
 * its group's B and C -- so N devices can each compute a range of heads of
 * one problem with no exchange (devotd.net page on the Mamba-2 cuTile forward
 * kernels, section 2: the state's independent parts are processed in
 * parallel).  Every pointer and size is that of ssd_forward for the WHOLE
 * problem (nheads heads); the call reads only the rows of its heads (and of
 * the B/C groups they use) and writes only their rows of y and final_state,
 * leaving the other heads' outputs untouched.  ssd_partition_heads gives a
 * balanced range per device.  The workspace is allocated as in ssd_forward,
 * sized for head_count heads.  Results equal ssd_forward's for those heads up
 * to rounding (the work is tiled for the call's head count).
 * Extra errors: SSD_ERR_INVALID_ARG if head_begin < 0, head_count < 1 or
 * head_begin + head_count > nheads.
 */
SSD_API int ssd_forward_heads(const void* x, const float* dt, const float* A, const void* B, const void* C,
                              const float* D, const float* init_state, int batch, int seqlen, int nheads,
                              int headdim, int ngroups, int dstate, int chunk_size, int head_begin, int head_count,
                              void* y, float* final_state, cudaStream_t stream);

/*
 * ssd_partition_heads -- the heads that part `part` of `nparts` (one per
 * device) computes with ssd_forward_heads: a contiguous range, the ranges of
 * all parts covering every head exactly once.  With at least as many B/C
 * groups as parts the ranges are whole groups, so a device reads only its own
 * groups' B and C; otherwise heads are split as evenly as possible in blocks
 * of two (one block never straddling a group boundary), and a part may get
 * no heads (*head_count == 0) when there are more parts than blocks.
 * Host-only; touches no device.  Returns SSD_ERR_INVALID_ARG for
 * non-positive sizes, nheads % ngroups != 0, part outside [0, nparts) or NULL
 * outputs, else SSD_OK.
 */
SSD_API int ssd_partition_heads(int nheads, int ngroups, int nparts, int part, int* head_begin, int* head_count);

/*
 * ssd_forward_noalloc -- ssd_forward with no memory allocation of any kind.
 * The pages describe no such variant; it exists for callers that must not
 * have the library allocate device memory during a call: code that has
 * already reserved the device's memory for its own allocator (so a pool of
 * the library's could not grow, or would compete with it), code that
 * accounts for every byte it places on the device, and latency-critical
 * loops where a pool that has to grow would stall the call.
 *
 * Arguments, layouts, ownership, results and errors are those of
 * ssd_forward.  Instead of a pool, the workspace lives in one fixed array of
 * SSD_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library's device image on
 * each device, so the library's footprint includes that array whether or not
 * this function is called.  The workspace of a call is about
 *     8 * batch * nheads * nchunks * chunk_size      (cumulative sums, dt)
 *   + 4 * batch * nspans * nheads * headdim * dstate (span states)
 *   + 4 * batch * nheads * nspans                    (span decays)
 *   + 4 * batch * seqlen * ngroups * dstate          (float16 B and C)
 * bytes, each part rounded up to 256 bytes, where nspans is the number of
 * chunk groups the library forms (about 1216 (batch, head, group) units);
 * a call that would need more returns SSD_ERR_SCRATCH_TOO_SMALL and launches
 * nothing -- use ssd_forward for such sizes (ssd_forward_plan reports the
 * exact figure beforehand).  For example batch 2,
 * seqlen 4096, nheads 64, dstate 128, chunk 256 needs 40 MiB and fits;
 * seqlen 65536, nheads 32, dstate 128 needs 85 MiB and does not.
 *
 * The first call on each device performs a one-time set-up with that device
 * current: it looks up the device address of the scratch array (and, like
 * every entry point, sets each kernel's shared-memory limit on first use).
 * Make that first call outside any stream capture.
 *
 * All calls on one device share the one scratch array.  Calls issued on the
 * same stream are ordered and safe; calls that may overlap on the device
 * (different streams, or host threads on different streams) race on the
 * scratch and give wrong results.  Nothing in the scratch needs to start at
 * zero: every call writes each part before reading it.
 */
SSD_API int ssd_forward_noalloc(const void* x, const float* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* init_state, int batch,
                        int seqlen, int nheads, int headdim, int ngroups, int dstate,
                        int chunk_size, void* y, float* final_state, cudaStream_t stream);

/*
 * ssd_backward -- gradients of a scalar loss through ssd_forward, given
 * dLoss/dy and dLoss/dfinal_state.  The pages describe no backward pass (they
 * only note that training speed depends on one); this is the reverse mode of
 * the recurrence ssd_forward computes, derived from it.  Per head h (group g),
 * with lam_t = dLoss/dstate after token t:
 *     lam_{L-1} = dfinal + C_{L-1} dy_{L-1}^T,   lam_t = exp(dt_{t+1} A) lam_{t+1} + C_t dy_t^T
 *     dx_t  = dt_t lam_t^T B_t + D dy_t
 *     dB_t  = sum over the group's heads of dt_t lam_t x_t
 *     dC_t  = sum over the group's heads of state_t dy_t
 *     ddt_t = A exp(dt_t A) <lam_t, state_{t-1}> + <lam_t, B_t x_t^T>
 *     dA    = sum over batch and tokens of dt_t exp(dt_t A) <lam_t, state_{t-1}>
 *     dD    = sum over batch, tokens and channels of x dy
 *     dinit = exp(dt_0 A) lam_0
 * computed in the forward's chunked form (blocks of 128 tokens, whatever
 * chunk_size is: the result does not depend on the chunking): a forward hop
 * for the state before every block, a reverse hop for the gradient flowing
 * into every block's end, then per (block, group) one pass over the group's
 * heads on tcgen05 tensor cores (every sum of the dt gradient kept inside a
 * block), and a fixed-order reduction of the per-block parts of dA and dD.
 * Operands of the products are float16 (as in ssd_forward), accumulation
 * float32; the hops read each block's own term as float16 and carry the
 * recurrence in float32.
 *
 * Inputs: as ssd_forward (x, B, C bf16; dt, A, D, init_state f32; D and
 * init_state nullable), dy (batch, seqlen, nheads, headdim) bf16, dfinal
 * (batch, nheads, headdim, dstate) f32 or NULL (= 0).  Outputs, all
 * caller-owned device memory, fully written:
 *     dx    (batch, seqlen, nheads, headdim)  bf16
 *     ddt   (batch, seqlen, nheads)           f32
 *     dA    (nheads)                          f32
 *     dB,dC (batch, seqlen, ngroups, dstate)  f32
 *     dD    (nheads) f32, or NULL (not computed)
 *     dinit (batch, nheads, headdim, dstate)  f32, or NULL (not computed)
 * x, B, C, dy, dx, dB, dC, init_state, dfinal and dinit 16-byte aligned; the
 * other pointers 4-byte aligned.  Supported: headdim 64, dstate 64 or 128,
 * otherwise the shape limits of ssd_forward (SSD_ERR_UNSUPPORTED).  The
 * workspace (about 3 x batch x nheads x headdim x dstate x 2 bytes per 128
 * tokens, plus float16 copies of B and C) is allocated stream-ordered from
 * the library's pool.  Deterministic: no atomics; dB and dC are summed over
 * a group's heads in a fixed order.  Errors: SSD_ERR_INVALID_ARG,
 * SSD_ERR_UNSUPPORTED, SSD_ERR_NO_MEMORY, SSD_ERR_CUDA; SSD_ERR_TIMEOUT and
 * SSD_ERR_RANGE through ssd_get_device_error, as for ssd_forward.
 */
SSD_API int ssd_backward(const void* x, const float* dt, const float* A, const void* B, const void* C,
                         const float* D, const float* init_state, const void* dy, const float* dfinal,
                         int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                         int chunk_size, void* dx, float* ddt, float* dA, float* dB, float* dC, float* dD,
                         float* dinit, cudaStream_t stream);

/*
 * ssd_forward_plan -- how ssd_forward and ssd_forward_noalloc split a
 * workload of these sizes, without touching device memory or launching
 * anything (a host-side query; no counterpart in the pages):
 *   span_chunks    chunks per span of the state stages (chunk_state runs
 *                  one CTA per span and few heads, state_passing hops over
 *                  spans): the shortest span of at most 64 chunks whose
 *                  chunk_state grid fits one CTA per multiprocessor, else
 *                  about eight waves of (batch, head, span) units;
 *   scan_step      spans per compute_out CTA (1, 2 or 4), chosen from the
 *                  current device's multiprocessor count (152 when no
 *                  device can be queried);
 *   noalloc_bytes  the workspace ssd_forward_noalloc would place in its
 *                  fixed scratch: the call fits when this is at most
 *                  SSD_NOALLOC_SCRATCH_BYTES (ssd_forward allocates about
 *                  as much from its pool).
 * Any output pointer may be NULL.  Returns the errors of ssd_forward's
 * shape checks (SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED), else SSD_OK.
 */
SSD_API int ssd_forward_plan(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                             int chunk_size, int* span_chunks, int* scan_step,
                             unsigned long long* noalloc_bytes);

/*
 * ssd_step -- one recurrent step of the selective state-space model for a
 * single new token of every sequence: the fixed-size-state mode of the model
 * (disconfirmai.com page, SSM/attention/RNN paragraph; readmex.ai page,
 * English excerpt: constant memory per token).  Per batch row b and head h,
 * g = h / (nheads / ngroups):
 *     a = exp(dt[b,h] * A[h])
 *     state[b,h,p,n] <- a * state[b,h,p,n] + dt[b,h] * B[b,g,n] * x[b,h,p]
 *     y[b,h,p] = sum_n C[b,g,n] * state[b,h,p,n] + D[h] * x[b,h,p]
 * i.e. ssd_forward over one token with init_state = final_state = state.
 *   x, y      (batch, nheads, headdim)   bfloat16 (2-byte aligned)
 *   dt        (batch, nheads)            float32
 *   A, D      (nheads)                   float32; D may be NULL (no skip term)
 *   B, C      (batch, ngroups, dstate)   bfloat16
 *   state     (batch, nheads, headdim, dstate) float32, 16-byte aligned; read
 *             and overwritten in place with the state after the token.
 * fp32 arithmetic throughout (exp is the accurate expf).  Supported shapes as
 * for ssd_forward (headdim 64, dstate 64/128/256/512).  Asynchronous on
 * `stream`; the same error behaviour as the other entry points.
 */
SSD_API int ssd_step(const void* x, const float* dt, const float* A, const void* B, const void* C,
                     const float* D, float* state, int batch, int nheads, int headdim, int ngroups, int dstate,
                     void* y, cudaStream_t stream);

/*
 * ssd_step_multi -- ntokens consecutive new tokens of every sequence in one
 * call: ssd_step applied ntokens times in order, with the state kept on chip
 * between the tokens, so the state is read and written once per call rather
 * than once per token.  Each token's arithmetic is that of ssd_step, so the
 * results equal ntokens ssd_step calls exactly.  It is the recurrence
 * itself (work linear in ntokens, no chunked matrix products): for short
 * bursts such as speculative or multi-token decoding; long prompts belong in
 * ssd_forward.  The readings are those of ssd_step (same pages):
 *   x, y      (batch, ntokens, nheads, headdim)  bfloat16 (2-byte aligned)
 *   dt        (batch, ntokens, nheads)           float32
 *   A, D      (nheads)                           float32; D may be NULL
 *   B, C      (batch, ntokens, ngroups, dstate)  bfloat16
 *   state     (batch, nheads, headdim, dstate)   float32, 16-byte aligned;
 *             read, then overwritten with the state after the last token.
 * These are ssd_forward's layouts with seqlen = ntokens and
 * init_state = final_state = state.  Errors as ssd_step, plus
 * SSD_ERR_INVALID_ARG for ntokens <= 0.
 */
SSD_API int ssd_step_multi(const void* x, const float* dt, const float* A, const void* B, const void* C,
                           const float* D, float* state, int batch, int ntokens, int nheads, int headdim,
                           int ngroups, int dstate, void* y, cudaStream_t stream);

/*
 * Input-side options of a whole Mamba-2 layer around the scan.  The pages
 * take dt as already positive and D as one weight per head; these are the
 * plainest reading of the steps a layer adds on either side, applied per
 * token and head in this order:
 *     dt <- dt + dt_bias[h]                    if dt_bias != NULL
 *     dt <- log(1 + exp(dt))                   if dt_softplus
 *     dt <- min(max(dt, dt_min), dt_max)       if dt_limit
 *     skip term D[h][p] * x[p]                 if D_per_channel (D is (nheads, headdim))
 *     y  <- y * z * sigmoid(z)                 if z != NULL (after the skip term)
 * z has x's layout, bfloat16, 16-byte aligned for ssd_forward_ex (2-byte for
 * ssd_step_ex); a per-channel D is 16-byte aligned for ssd_forward_ex.
 * dt_bias is (nheads) float32.  A zero-filled struct (or a
 * NULL pointer) selects none of them.  The options change only the inputs
 * and the output: the carried state is never gated.
 */
typedef struct ssd_input_options {
    const float* dt_bias;
    int dt_softplus;
    int dt_limit;
    float dt_min;
    float dt_max;
    int D_per_channel;
    const void* z;
} ssd_input_options;

/*
 * ssd_forward_ex -- ssd_forward with the input-side options above (options
 * may be NULL: then it is ssd_forward).  The dt transform is applied where
 * dt is first read (chunk_cumsum), so every later stage sees the effective
 * dt.  A per-channel D enters compute_out as one more tensor-core product,
 * Y += X diag(D), so D is rounded to float16 there (11 significant bits; D
 * beyond the float16 range saturates); the z gate is applied in
 * compute_out's epilogue, in fp32.
 * Extra errors: SSD_ERR_INVALID_ARG if dt_limit is set with dt_min > dt_max
 * or a NaN bound, if z or a per-channel D is not 16-byte aligned, or dt_bias
 * not 4-byte aligned.
 */
SSD_API int ssd_forward_ex(const void* x, const float* dt, const float* A, const void* B, const void* C,
                           const float* D, const float* init_state, int batch, int seqlen, int nheads,
                           int headdim, int ngroups, int dstate, int chunk_size,
                           const ssd_input_options* options, void* y, float* final_state,
                           cudaStream_t stream);

/*
 * ssd_step_ex -- ssd_step with the input-side options (NULL: ssd_step).
 * With D_per_channel, D is (nheads, headdim); z is (batch, nheads, headdim)
 * bfloat16.  Errors as ssd_step plus those of ssd_forward_ex's options.
 */
SSD_API int ssd_step_ex(const void* x, const float* dt, const float* A, const void* B, const void* C,
                        const float* D, float* state, int batch, int nheads, int headdim, int ngroups,
                        int dstate, const ssd_input_options* options, void* y, cudaStream_t stream);

/*
 * ssd_get_device_error -- reads and clears the library's device error words
 * on the current device (synchronizes with the device).  Returns SSD_OK;
 * SSD_ERR_TIMEOUT if a kernel's bounded wait gave up since the last read
 * (the kernel then skipped the rest of its work and returned, so the outputs
 * of that call are incomplete while the device stays usable); otherwise
 * SSD_ERR_RANGE if a value converted to a float16 tensor-core operand was
 * outside float16's finite range since the last read; or SSD_ERR_CUDA if the
 * read itself failed.
 */
SSD_API int ssd_get_device_error(void);

/*
 * Test hooks of the failure path (no counterpart in the pages; process-wide,
 * they affect every later launch until reset).
 * ssd_debug_set_wait_limit_ns(ns) sets the time after which a pipeline wait
 * inside the tensor-core kernels (chunk_state, chunk_scan) gives up; 0
 * restores the default of one second.  The teardown drains that let every
 * copy and product already issued complete before a kernel releases shared
 * memory and TMEM keep their own one-second limit.
 * ssd_debug_stall(kinds) makes every later launch of the selected kernel
 * kinds (bit k = kind k of ssd_kernel_name; 0 turns it off) first wait on a
 * barrier that nothing completes: the wait runs out after the wait limit,
 * the kernel abandons its work and returns, and ssd_get_device_error()
 * reports SSD_ERR_TIMEOUT.  A stalled call's outputs are incomplete.
 * Both return SSD_OK.
 */
SSD_API int ssd_debug_set_wait_limit_ns(unsigned long long ns);
SSD_API int ssd_debug_stall(int kinds);

/*
 * Profiling counters (host side, process-wide, not thread-safe).
 * ssd_profile_enable(kinds) makes every later launch of a selected kernel
 * kind record a CUDA event pair around itself on the launch stream: `kinds`
 * is a bit mask over the kinds of ssd_kernel_name (bit k selects kind k),
 * -1 selects all and 0 turns profiling off.  Each event pair adds a few
 * microseconds between launches, so a timed loop can select only the kernel
 * it needs.  ssd_profile_read() waits for those
 * events and returns, per kernel kind (see ssd_kernel_name), the summed
 * device time in milliseconds and the launch count since the last reset.
 * ssd_launch_count() counts every kernel the library has launched since load
 * (profiling enabled or not).
 */
SSD_API int ssd_profile_enable(int kinds);
SSD_API int ssd_profile_reset(void);
SSD_API int ssd_profile_read(float* total_ms, int* launches, int max_kinds, int* n_kinds);
SSD_API const char* ssd_kernel_name(int kind);
SSD_API long long ssd_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
