// ssd_api.cu -- the C ABI: argument validation, workspace, launch sequencing,
// device error word and profiling counters.  Every exported function is
// declared (and documented) in include/ssd.h.
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <array>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "common.cuh"

namespace ssd {

// ------------------------------------------------------------ profiling
namespace {

struct EventPair {
    int kind;
    cudaEvent_t start, stop;
};

std::mutex g_prof_mu;
unsigned g_prof_mask = 0;  // bit k: launches of kernel kind k record an event pair
std::vector<EventPair> g_prof_open;   // recorded, not yet read
std::vector<cudaEvent_t> g_prof_free; // reusable events
double g_prof_ms[kNumKinds];
int g_prof_count[kNumKinds];
long long g_launches = 0;
EventPair g_pending = {-1, nullptr, nullptr};

cudaEvent_t take_event() {
    if (!g_prof_free.empty()) {
        cudaEvent_t e = g_prof_free.back();
        g_prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

const char* const kKindNames[kNumKinds] = {"chunk_cumsum", "chunk_state", "state_passing", "chunk_scan",
                                           "bc_to_f16", "step", "bwd_chunk", "bwd_reduce"};

}  // namespace

void launch_begin(int kind, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_pending.kind = -1;
    if (kind < 0 || kind >= 32 || !((g_prof_mask >> kind) & 1u)) return;
    cudaEvent_t a = take_event(), b = take_event();
    if (a == nullptr || b == nullptr) return;
    cudaEventRecord(a, s);
    g_pending = {kind, a, b};
}

int launch_end(int kind, cudaStream_t s) {
    const cudaError_t e = cudaGetLastError();
    std::lock_guard<std::mutex> lk(g_prof_mu);
    ++g_launches;
    if (g_pending.kind == kind) {
        cudaEventRecord(g_pending.stop, s);
        g_prof_open.push_back(g_pending);
        g_pending.kind = -1;
    }
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

int ensure_smem_limit(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::vector<std::pair<const void*, int>> done;  // (kernel, device)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    for (auto& e : done)
        if (e.first == kernel && e.second == dev) return SSD_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return SSD_ERR_CUDA;
    done.emplace_back(kernel, dev);
    return SSD_OK;
}

}  // namespace ssd

using namespace ssd;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dstate(int n) { return n == 64 || n == 128 || n == 256 || n == 512; }
bool supported_chunk(int q) { return q == 64 || q == 128 || q == 256; }

// Shape validation shared by the entry points.  Returns SSD_OK or an error.
int check_dims(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk_size) {
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 ||
        chunk_size <= 0)
        return SSD_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (headdim != 64 || !supported_dstate(dstate) || !supported_chunk(chunk_size)) return SSD_ERR_UNSUPPORTED;
    // element counts must fit the kernels' 64-bit offsets and grid limits
    const int64_t nchunks = ((int64_t)seqlen + chunk_size - 1) / chunk_size;
    if (nchunks > 65535 * 64 || batch > 65535 || nheads > 4096) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// Validates the input-side options and splits them into the dt transform
// (chunk_cumsum / step) and the output options (compute_out's epilogue / step).
// `rows16`: z and a per-channel D are read in 16-byte pieces (ssd_forward_ex).
int read_options(const ssd_input_options* o, const float* D, bool rows16, DtOpts* dto, OutOpts* oo) {
    *dto = DtOpts();
    *oo = OutOpts();
    if (o == nullptr) return SSD_OK;
    if (o->dt_bias != nullptr && (reinterpret_cast<uintptr_t>(o->dt_bias) & 3u)) return SSD_ERR_INVALID_ARG;
    if (o->dt_limit && !(o->dt_min <= o->dt_max)) return SSD_ERR_INVALID_ARG;  // also rejects a NaN bound
    if (o->z != nullptr && (rows16 ? !aligned16(o->z) : (reinterpret_cast<uintptr_t>(o->z) & 1u)))
        return SSD_ERR_INVALID_ARG;
    if (o->D_per_channel && D != nullptr && rows16 && !aligned16(D)) return SSD_ERR_INVALID_ARG;
    dto->bias = o->dt_bias;
    dto->softplus = o->dt_softplus != 0;
    dto->limit = o->dt_limit != 0;
    dto->lo = o->dt_min;
    dto->hi = o->dt_max;
    if (o->D_per_channel) oo->Dp = D;
    oo->z = static_cast<const __nv_bfloat16*>(o->z);
    return SSD_OK;
}

Dims make_dims(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk_size) {
    Dims d;
    d.batch = batch;
    d.seqlen = seqlen;
    d.nheads = nheads;
    d.headdim = headdim;
    d.ngroups = ngroups;
    d.dstate = dstate;
    d.chunk_size = chunk_size;
    d.nchunks = (seqlen + chunk_size - 1) / chunk_size;
    d.head0 = 0;
    d.hcount = nheads;
    return d;
}

}  // namespace

// device error words: [0] the code of a bounded wait that gave up, [1] the float16 range flag
__device__ int g_ssd_device_error[2] = {0, 0};

namespace {

// Limit of the kernels' pipeline waits and the kernel kinds whose launches take the stall hook
// (ssd_debug_set_wait_limit_ns, ssd_debug_stall).
std::atomic<unsigned long long> g_wait_ns{1000000000ull};
std::atomic<int> g_stall_kinds{0};

// Device address of g_ssd_device_error on the current device (cached per device).
int* device_error_ptr() {
    static std::mutex mu;
    static int* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 64 && cache[dev] != nullptr) return cache[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ssd_device_error) != cudaSuccess) return nullptr;
    if (dev < 64) cache[dev] = static_cast<int*>(p);
    return static_cast<int*>(p);
}

// Stream-ordered workspace from a library-owned pool per device that keeps
// freed memory cached (release threshold = max), so repeated calls neither
// map nor unmap device memory.
cudaMemPool_t workspace_pool() {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (pools[dev] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        pools[dev] = p;
    }
    return pools[dev];
}

// Failure-handling arguments of one launch of kernel kind `kind`.
Ctl make_ctl(int* err, int kind) {
    Ctl c;
    c.err = err;
    c.wait_ns = g_wait_ns.load();
    c.stall = (g_stall_kinds.load() >> kind) & 1;
    return c;
}

int workspace_alloc(void** ptr, size_t bytes, cudaStream_t s) {
    cudaMemPool_t p = workspace_pool();
    if (p == nullptr || cudaMallocFromPoolAsync(ptr, bytes, p, s) != cudaSuccess) {
        cudaGetLastError();
        return SSD_ERR_NO_MEMORY;
    }
    return SSD_OK;
}

int device_sms();

// Chunks per span for ssd_forward: about eight waves of 152 CTAs over
// (batch, head, span), so the span-level intermediates stay small while
// every SM stays busy -- or, when a span of at most 64 chunks makes chunk_state's grid
// (batch, heads / heads per CTA, spans) fit one CTA per SM, the shortest such span: chunk_state then
// runs its CTAs all at once with twice the stages in flight, and the hop has fewer spans to cross.
int forward_span_chunks(const Dims& d) {
    const int64_t units = (int64_t)d.batch * d.hcount * d.nchunks;
    int64_t k = (units + 1215) / 1216;
    if (k < 1) k = 1;
    if (k > 64) k = 64;
    if (k > d.nchunks) k = d.nchunks;
    const int64_t rows = (int64_t)d.batch * (d.hcount / chunk_state_heads_per_cta(d));
    const int sms = device_sms();
    for (int64_t k1 = k; k1 <= 64 && k1 <= d.nchunks; ++k1)
        if (rows * ceil_div64(d.nchunks, k1) <= sms) return (int)k1;
    return (int)k;
}

// Multiprocessor count of the current device (cached per device).
int device_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lk(mu);
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

// Makespan, in 128-token sub-block times, of one chunk_scan launch over `sms` SMs (one CTA per
// SM) when CTAs start in launch order (head fastest, then span, then batch) on the first free SM.
// A CTA costs its sub-blocks plus a fixed pipeline fill and drain of about 1.2 sub-block times
// (fitted to CUDA-event times of chunk_scan on GB300 at several span lengths).
double scan_makespan(int64_t rows_per_batch, int batch, int nchunks, int chunk_size, int span2, int sms) {
    const double fill = 1.2;
    const int ns = ceil_div(nchunks, span2);
    const double full = std::ceil((double)span2 * chunk_size / 128.0);
    const double last = std::ceil((double)(nchunks - (ns - 1) * span2) * chunk_size / 128.0);
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < sms; ++i) free_at.push(0.0);
    double end = 0.0;
    for (int b = 0; b < batch; ++b)
        for (int sp = 0; sp < ns; ++sp)
            for (int64_t r = 0; r < rows_per_batch; ++r) {
                const double t = free_at.top() + fill + (sp == ns - 1 ? last : full);
                free_at.pop();
                free_at.push(t);
                if (t > end) end = t;
            }
    return end;
}

// Span-start states per chunk_scan span: chunk_scan walks spans of `span` * step chunks
// (step in {1, 2, 4}), each from every step-th span-start state, so there are fewer, longer
// CTAs and less pipeline fill and drain per sub-block.  The step with the shortest estimated
// makespan wins (by at least 0.5%); decided once per shape.
// A CTA of the paired kernel covers two heads, so its rows are head pairs.
int forward_scan_step(const Dims& d, int span, const OutOpts& oo) {
    static std::mutex mu;
    static std::map<std::array<int64_t, 6>, int> cache;
    const int sms = device_sms();
    const bool pair = chunk_scan_pair_supported(d, oo);
    const std::array<int64_t, 6> key = {d.batch, d.hcount, d.nchunks, span, sms, pair ? 1 : 0};
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int64_t rows = pair ? d.hcount / 2 : d.hcount;
    int best = 1;
    double best_t = scan_makespan(rows, d.batch, d.nchunks, d.chunk_size, span, sms);
    for (int m = 2; m <= 4; m *= 2) {
        if ((int64_t)span * m > d.nchunks) break;
        // one wave that leaves SMs idle can still beat two fuller ones: the estimate decides
        const double t = scan_makespan(rows, d.batch, d.nchunks, d.chunk_size, span * m, sms);
        if (t < best_t * 0.995) {
            best = m;
            best_t = t;
        }
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = best;
    return best;
}

// CTAs per (block, group) of the backward kernel: the heads of a group split into S slices (a cluster
// whose partial dB / dC are added on chip).  With one CTA per SM, S is the value of 1, 2, 4 (dividing
// the heads per group) with the smallest estimated makespan, waves x (heads per CTA + 1): the 1 is
// the per-CTA setup and the cluster's final sum, about one head's time.
int bwd_slices(const Dims& d) {
    const int sms = device_sms();
    const int hpg = d.nheads / d.ngroups;
    int best = 1;
    double best_t = 0.0;
    for (int S = 1; S <= 4; S *= 2) {
        if (hpg % S != 0) break;
        const int64_t ctas = (int64_t)d.nchunks * d.ngroups * S * d.batch;
        const double t = (double)((ctas + sms - 1) / sms) * (hpg / S + 1);
        if (S == 1 || t < best_t) {
            best = S;
            best_t = t;
        }
    }
    return best;
}

}  // namespace

// ---------------------------------------------------------------- fixed scratch
// Scratch for ssd_forward_noalloc: a fixed array in the library's own device
// image, so that call needs no allocation at all.  Every call on a device uses
// the same bytes.  Nothing in it has to start at zero: each region is fully
// written by an earlier kernel of the same call before any kernel reads it.
static __device__ __align__(256) unsigned char g_ssd_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the fixed scratch on the current device, looked up once
// per device (with that device current) and cached.
unsigned char* noalloc_scratch_ptr() {
    static std::mutex mu;
    static unsigned char* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == nullptr) {
        unsigned char* p = nullptr;
        if (cudaGetSymbolAddress((void**)&p, g_ssd_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = p;
    }
    return cache[dev];
}

size_t round256(size_t bytes) { return (bytes + 255) & ~(size_t)255; }

// Byte offsets of ssd_forward_noalloc's workspace parts inside the fixed scratch (each part starts
// on a 256-byte boundary): dA_cumsum, dt rows, span states, span decays, float16 B, float16 C.
struct NoallocLayout {
    size_t off_dtt, off_S, off_dec, off_B16, off_C16, need;
};

NoallocLayout noalloc_layout(const Dims& d, int span) {
    const int nspans = ceil_div(d.nchunks, span);
    const size_t ncq = (size_t)d.batch * d.hcount * d.nchunks * d.chunk_size;
    const size_t nst = (size_t)d.batch * nspans * d.hcount * d.headdim * d.dstate;
    const size_t ndec = (size_t)d.batch * d.hcount * nspans;
    const size_t nbc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;
    NoallocLayout l;
    l.off_dtt = round256(ncq * sizeof(float));
    l.off_S = l.off_dtt + round256(ncq * sizeof(float));
    l.off_dec = l.off_S + round256(nst * sizeof(float));
    l.off_B16 = l.off_dec + round256(ndec * sizeof(float));
    l.off_C16 = l.off_B16 + round256(nbc * sizeof(__half));
    l.need = l.off_C16 + round256(nbc * sizeof(__half));
    return l;
}

// The four stages of one forward over the call's heads (d.head0, d.hcount), with the workspace parts
// given: dA_cumsum and dt rows (b, hcount, nc, Q), span states (b, nspans, hcount, P, N), span decays
// (b, hcount, nspans), float16 B and C (the caller's layout; the groups of the call's heads written).
int run_forward(const Dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                const float* D, const float* init_state, void* y, float* final_state, float* cs, float* dtt, float* S,
                float* dec, __half* B16, __half* C16, int* err, cudaStream_t stream, const DtOpts& dto,
                const OutOpts& oo) {
    const int span = forward_span_chunks(d);
    const int nspans = ceil_div(d.nchunks, span);
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    int r = launch_chunk_cumsum_bc(dt, A, d, cs, dtt, static_cast<const __nv_bfloat16*>(B),
                                   static_cast<const __nv_bfloat16*>(C), B16, C16, err, stream, dto);
    if (r == SSD_OK)
        r = launch_chunk_state_span(xb, B16, dtt, cs, span, d, S, dec, make_ctl(err, kKindChunkState), stream);
    // span-level hop, in place: S becomes the span-start states
    if (r == SSD_OK) r = launch_state_passing_steps(S, dec, 1, nspans, init_state, d, nspans, S, final_state, stream);
    if (r == SSD_OK)
        r = launch_chunk_scan_span(xb, B16, C16, dtt, cs, D, S, span, d, static_cast<__nv_bfloat16*>(y),
                                   make_ctl(err, kKindChunkScan), stream, oo, forward_scan_step(d, span, oo));
    return r;
}

// Validation shared by the forward entry points (pointers, shapes, alignment).
int check_forward(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                  const float* init_state, int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                  int chunk_size, const void* y, const float* final_state) {
    if (!x || !dt || !A || !B || !C || !y) return SSD_ERR_INVALID_ARG;
    const int r = check_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    if (r != SSD_OK) return r;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(y) || ((uintptr_t)dt & 3u) ||
        ((uintptr_t)A & 3u) || (D && ((uintptr_t)D & 3u)) || (init_state && !aligned16(init_state)) ||
        (final_state && !aligned16(final_state)))
        return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

// Forward over the heads of d with a stream-ordered workspace from the library's pool.
int forward_pooled(const Dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
                   const float* D, const float* init_state, void* y, float* final_state, cudaStream_t stream,
                   const DtOpts& dto, const OutOpts& oo) {
    int* err = device_error_ptr();
    if (err == nullptr) return SSD_ERR_CUDA;
    const int span = forward_span_chunks(d);
    const int nspans = ceil_div(d.nchunks, span);
    const size_t ncq = (size_t)d.batch * d.hcount * d.nchunks * d.chunk_size;
    const size_t nst = (size_t)d.batch * nspans * d.hcount * d.headdim * d.dstate;
    const size_t ndec = ((size_t)d.batch * d.hcount * nspans + 3) & ~(size_t)3;
    const size_t nbc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;  // multiple of 64
    const size_t bytes = (2 * ncq + nst + ndec) * sizeof(float) + 2 * nbc * sizeof(__half);
    void* ws = nullptr;
    if (workspace_alloc(&ws, bytes, stream) != SSD_OK) return SSD_ERR_NO_MEMORY;
    float* cs = static_cast<float*>(ws);
    float* dtt = cs + ncq;
    float* S = dtt + ncq;
    float* dec = S + nst;
    __half* B16 = reinterpret_cast<__half*>(dec + ndec);
    __half* C16 = B16 + nbc;
    int r = run_forward(d, x, dt, A, B, C, D, init_state, y, final_state, cs, dtt, S, dec, B16, C16, err, stream, dto,
                        oo);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && r == SSD_OK) r = SSD_ERR_CUDA;
    return r;
}

}  // namespace

extern "C" {

const char* ssd_status_string(int status) {
    switch (status) {
        case SSD_OK: return "SSD_OK: success";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: null pointer, non-positive size, misalignment or bad grouping";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: shape outside the implemented set";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA call or kernel launch failed";
        case SSD_ERR_NO_MEMORY: return "SSD_ERR_NO_MEMORY: workspace allocation failed";
        case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded device-side wait gave up";
        case SSD_ERR_RANGE:
            return "SSD_ERR_RANGE: a value converted to a float16 tensor-core operand exceeded float16's range "
                   "(|v| > 65504); that call's results are not reliable";
        case SSD_ERR_SCRATCH_TOO_SMALL:
            return "SSD_ERR_SCRATCH_TOO_SMALL: the workload needs more than the fixed scratch of ssd_forward_noalloc "
                   "(SSD_NOALLOC_SCRATCH_BYTES); use ssd_forward";
        default: return "unknown ssd status";
    }
}

int ssd_chunk_cumsum(const float* dt, const float* A, int batch, int seqlen, int nheads, int chunk_size,
                     float* dA_cumsum, float* dt_t, cudaStream_t stream) {
    if (!dt || !A || !dA_cumsum || !dt_t) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || chunk_size <= 0) return SSD_ERR_INVALID_ARG;
    if (!aligned16(dA_cumsum) || !aligned16(dt_t) || ((uintptr_t)dt & 3u) || ((uintptr_t)A & 3u))
        return SSD_ERR_INVALID_ARG;
    if (!supported_chunk(chunk_size)) return SSD_ERR_UNSUPPORTED;
    const int64_t nchunks = ((int64_t)seqlen + chunk_size - 1) / chunk_size;
    if (nchunks > 2147483647LL || batch > 65535 || nheads > 65535 * 8) return SSD_ERR_UNSUPPORTED;
    Dims d = make_dims(batch, seqlen, nheads, 64, 1, 64, chunk_size);
    return launch_chunk_cumsum(dt, A, d, dA_cumsum, dt_t, stream);
}

int ssd_chunk_state(const void* x, const void* B, const float* dt_t, const float* dA_cumsum, int batch,
                    int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk_size,
                    float* chunk_states, cudaStream_t stream) {
    if (!x || !B || !dt_t || !dA_cumsum || !chunk_states) return SSD_ERR_INVALID_ARG;
    int r = check_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    if (r != SSD_OK) return r;
    if (!aligned16(x) || !aligned16(B) || !aligned16(dt_t) || !aligned16(dA_cumsum) || !aligned16(chunk_states))
        return SSD_ERR_INVALID_ARG;
    Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    int* err = device_error_ptr();
    if (err == nullptr) return SSD_ERR_CUDA;
    // stream-ordered float16 copy of B for the tensor-core products
    const size_t nbc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;
    void* ws = nullptr;
    if (workspace_alloc(&ws, nbc * sizeof(__half), stream) != SSD_OK) return SSD_ERR_NO_MEMORY;
    __half* B16 = static_cast<__half*>(ws);
    r = launch_bc_to_f16(static_cast<const __nv_bfloat16*>(B), nullptr, d, B16, nullptr, err, stream);
    if (r == SSD_OK)
        r = launch_chunk_state_span(static_cast<const __nv_bfloat16*>(x), B16, dt_t, dA_cumsum, 1, d, chunk_states,
                                    nullptr, make_ctl(err, kKindChunkState), stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && r == SSD_OK) r = SSD_ERR_CUDA;
    return r;
}

int ssd_state_passing(const float* chunk_states, const float* dA_cumsum, const float* init_state, int batch,
                      int nchunks, int nheads, int headdim, int dstate, int chunk_size, float* states,
                      float* final_state, cudaStream_t stream) {
    if (!chunk_states || !dA_cumsum || !states) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || nchunks <= 0 || nheads <= 0 || headdim <= 0 || dstate <= 0 || chunk_size <= 0)
        return SSD_ERR_INVALID_ARG;
    if (headdim != 64 || !supported_dstate(dstate) || !supported_chunk(chunk_size)) return SSD_ERR_UNSUPPORTED;
    if (batch > 65535 || nheads > 65535) return SSD_ERR_UNSUPPORTED;
    if (!aligned16(chunk_states) || !aligned16(states) || ((uintptr_t)dA_cumsum & 3u) ||
        (init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
        return SSD_ERR_INVALID_ARG;
    Dims d = make_dims(batch, nchunks * chunk_size, nheads, headdim, 1, dstate, chunk_size);
    d.nchunks = nchunks;
    return launch_state_passing(chunk_states, dA_cumsum, init_state, d, states, final_state, stream);
}

int ssd_chunk_scan(const void* x, const void* B, const void* C, const float* dt_t, const float* dA_cumsum,
                   const float* D, const float* states, int batch, int seqlen, int nheads, int headdim,
                   int ngroups, int dstate, int chunk_size, void* y, cudaStream_t stream) {
    if (!x || !B || !C || !dt_t || !dA_cumsum || !states || !y) return SSD_ERR_INVALID_ARG;
    int r = check_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    if (r != SSD_OK) return r;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(y) || !aligned16(dt_t) ||
        !aligned16(dA_cumsum) || !aligned16(states) || (D && ((uintptr_t)D & 3u)))
        return SSD_ERR_INVALID_ARG;
    Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    int* err = device_error_ptr();
    if (err == nullptr) return SSD_ERR_CUDA;
    // stream-ordered float16 copies of B and C for the tensor-core products
    const size_t nbc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;
    void* ws = nullptr;
    if (workspace_alloc(&ws, 2 * nbc * sizeof(__half), stream) != SSD_OK) return SSD_ERR_NO_MEMORY;
    __half* B16 = static_cast<__half*>(ws);
    __half* C16 = B16 + nbc;
    r = launch_bc_to_f16(static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), d, B16, C16,
                         err, stream);
    if (r == SSD_OK)
        r = launch_chunk_scan_span(static_cast<const __nv_bfloat16*>(x), B16, C16, dt_t, dA_cumsum, D, states, 1, d,
                                   static_cast<__nv_bfloat16*>(y), make_ctl(err, kKindChunkScan), stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && r == SSD_OK) r = SSD_ERR_CUDA;
    return r;
}

int ssd_forward(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                const float* init_state, int batch, int seqlen, int nheads, int headdim, int ngroups,
                int dstate, int chunk_size, void* y, float* final_state, cudaStream_t stream) {
    return ssd_forward_ex(x, dt, A, B, C, D, init_state, batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size,
                          nullptr, y, final_state, stream);
}

int ssd_forward_ex(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                   const float* init_state, int batch, int seqlen, int nheads, int headdim, int ngroups,
                   int dstate, int chunk_size, const ssd_input_options* options, void* y, float* final_state,
                   cudaStream_t stream) {
    int r = check_forward(x, dt, A, B, C, D, init_state, batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size,
                          y, final_state);
    if (r != SSD_OK) return r;
    DtOpts dto;
    OutOpts oo;
    r = read_options(options, D, true, &dto, &oo);
    if (r != SSD_OK) return r;
    const Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    return forward_pooled(d, x, dt, A, B, C, D, init_state, y, final_state, stream, dto, oo);
}

int ssd_forward_heads(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                      const float* init_state, int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                      int chunk_size, int head_begin, int head_count, void* y, float* final_state,
                      cudaStream_t stream) {
    int r = check_forward(x, dt, A, B, C, D, init_state, batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size,
                          y, final_state);
    if (r != SSD_OK) return r;
    if (head_begin < 0 || head_count < 1 || head_begin > nheads - head_count) return SSD_ERR_INVALID_ARG;
    Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    d.head0 = head_begin;
    d.hcount = head_count;
    return forward_pooled(d, x, dt, A, B, C, D, init_state, y, final_state, stream, DtOpts(), OutOpts());
}

int ssd_partition_heads(int nheads, int ngroups, int nparts, int part, int* head_begin, int* head_count) {
    if (nheads <= 0 || ngroups <= 0 || nheads % ngroups != 0 || nparts <= 0 || part < 0 || part >= nparts ||
        !head_begin || !head_count)
        return SSD_ERR_INVALID_ARG;
    const int hpg = nheads / ngroups;
    int b = 0, e = 0;
    if (ngroups >= nparts) {
        // whole groups: part p takes groups [floor(p G / n), floor((p + 1) G / n))
        b = (int)((int64_t)part * ngroups / nparts) * hpg;
        e = (int)((int64_t)(part + 1) * ngroups / nparts) * hpg;
    } else {
        // fewer groups than parts: split heads evenly, in blocks of two heads where the count allows
        // (compute_out then keeps two heads per CTA), never a block across a group boundary
        const int unit = (hpg % 2 == 0) ? 2 : 1;
        const int nunits = nheads / unit;
        b = (int)((int64_t)part * nunits / nparts) * unit;
        e = (int)((int64_t)(part + 1) * nunits / nparts) * unit;
    }
    *head_begin = b;
    *head_count = e - b;
    return SSD_OK;
}

int ssd_forward_noalloc(const void* x, const float* dt, const float* A, const void* B, const void* C,
                        const float* D, const float* init_state, int batch, int seqlen, int nheads, int headdim,
                        int ngroups, int dstate, int chunk_size, void* y, float* final_state, cudaStream_t stream) {
    int r = check_forward(x, dt, A, B, C, D, init_state, batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size,
                          y, final_state);
    if (r != SSD_OK) return r;
    const Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    const int span = forward_span_chunks(d);
    // the same regions as ssd_forward, each starting on a 256-byte boundary
    const NoallocLayout l = noalloc_layout(d, span);
    if (l.need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_SCRATCH_TOO_SMALL;
    int* err = device_error_ptr();
    unsigned char* ws = noalloc_scratch_ptr();
    if (err == nullptr || ws == nullptr) return SSD_ERR_CUDA;
    return run_forward(d, x, dt, A, B, C, D, init_state, y, final_state, reinterpret_cast<float*>(ws),
                       reinterpret_cast<float*>(ws + l.off_dtt), reinterpret_cast<float*>(ws + l.off_S),
                       reinterpret_cast<float*>(ws + l.off_dec), reinterpret_cast<__half*>(ws + l.off_B16),
                       reinterpret_cast<__half*>(ws + l.off_C16), err, stream, DtOpts(), OutOpts());
}

int ssd_forward_plan(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk_size,
                     int* span_chunks, int* scan_step, unsigned long long* noalloc_bytes) {
    const int r = check_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    if (r != SSD_OK) return r;
    const Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    const int span = forward_span_chunks(d);
    if (span_chunks != nullptr) *span_chunks = span;
    if (scan_step != nullptr) *scan_step = forward_scan_step(d, span, OutOpts());
    if (noalloc_bytes != nullptr) *noalloc_bytes = (unsigned long long)noalloc_layout(d, span).need;
    return SSD_OK;
}

int ssd_backward(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                 const float* init_state, const void* dy, const float* dfinal, int batch, int seqlen, int nheads,
                 int headdim, int ngroups, int dstate, int chunk_size, void* dx, float* ddt, float* dA, float* dB,
                 float* dC, float* dD, float* dinit, cudaStream_t stream) {
    if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC) return SSD_ERR_INVALID_ARG;
    int r = check_dims(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size);
    if (r != SSD_OK) return r;
    if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(dy) || !aligned16(dx) || !aligned16(dB) ||
        !aligned16(dC) || ((uintptr_t)dt & 3u) || ((uintptr_t)A & 3u) || ((uintptr_t)ddt & 3u) ||
        ((uintptr_t)dA & 3u) || (D && ((uintptr_t)D & 3u)) || (dD && ((uintptr_t)dD & 3u)) ||
        (init_state && !aligned16(init_state)) || (dfinal && !aligned16(dfinal)) || (dinit && !aligned16(dinit)))
        return SSD_ERR_INVALID_ARG;
    // the backward works in blocks of kBwdBlock tokens whatever chunk_size is (the result does not depend
    // on the chunking)
    const Dims d = make_dims(batch, seqlen, nheads, headdim, ngroups, dstate, kBwdBlock);
    if (!bwd_supported(d)) return SSD_ERR_UNSUPPORTED;
    int* err = device_error_ptr();
    if (err == nullptr) return SSD_ERR_CUDA;
    const size_t nrow = (size_t)d.batch * d.nheads * d.nchunks * kBwdBlock;        // cs and dt rows
    const size_t nst = (size_t)d.batch * d.nchunks * d.nheads * d.headdim * d.dstate;  // per-block states
    const size_t npart = ((size_t)d.batch * d.nheads * d.nchunks + 3) & ~(size_t)3;  // per-block partial sums
    const size_t nbc = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;  // multiple of 64
    const size_t bytes = (2 * nrow + 2 * npart) * sizeof(float) + (3 * nst + 2 * nbc) * sizeof(__half);
    void* ws = nullptr;
    if (workspace_alloc(&ws, bytes, stream) != SSD_OK) return SSD_ERR_NO_MEMORY;
    float* cs = static_cast<float*>(ws);
    float* dtt = cs + nrow;
    float* dap = dtt + nrow;
    float* xdy = dap + npart;
    __half* h0 = reinterpret_cast<__half*>(xdy + npart);  // block-start states (float16)
    __half* mu = h0 + nst;                                // block-end gradients (float16)
    __half* S16 = mu + nst;  // the blocks' own states, then their own reverse-time terms (float16; the hops add in f32)
    __half* B16 = S16 + nst;
    __half* C16 = B16 + nbc;
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* dyb = static_cast<const __nv_bfloat16*>(dy);
    // forward hop: the state before every block
    r = launch_chunk_cumsum_bc(dt, A, d, cs, dtt, static_cast<const __nv_bfloat16*>(B),
                               static_cast<const __nv_bfloat16*>(C), B16, C16, err, stream);
    if (r == SSD_OK)
        r = launch_chunk_state_span(xb, B16, dtt, cs, 1, d, nullptr, nullptr, make_ctl(err, kKindChunkState), stream,
                                    S16);
    if (r == SSD_OK)
        r = launch_state_passing_steps(nullptr, cs + (kBwdBlock - 1), kBwdBlock, (int64_t)d.nchunks * kBwdBlock,
                                       init_state, d, d.nchunks, nullptr, nullptr, stream, 0, h0, err, S16);
    // reverse hop: the gradient flowing into the state after every block, and dinit
    if (r == SSD_OK)
        r = launch_chunk_state_rev(dyb, C16, dtt, cs, d, nullptr, make_ctl(err, kKindChunkState), stream, S16);
    if (r == SSD_OK)
        r = launch_state_passing_steps(nullptr, cs + (kBwdBlock - 1), kBwdBlock, (int64_t)d.nchunks * kBwdBlock,
                                       dfinal, d, d.nchunks, nullptr, dinit, stream, 1, mu, err, S16);
    if (r == SSD_OK)
        r = launch_bwd_chunk(xb, dyb, B16, C16, cs, dtt, A, D, h0, mu, d, static_cast<__nv_bfloat16*>(dx), ddt, dB, dC,
                             dap, xdy, make_ctl(err, kKindBwdChunk), stream, bwd_slices(d));
    if (r == SSD_OK) r = launch_bwd_reduce(dap, xdy, d, dA, dD, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && r == SSD_OK) r = SSD_ERR_CUDA;
    return r;
}

int ssd_step(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
             float* state, int batch, int nheads, int headdim, int ngroups, int dstate, void* y,
             cudaStream_t stream) {
    return ssd_step_ex(x, dt, A, B, C, D, state, batch, nheads, headdim, ngroups, dstate, nullptr, y, stream);
}

int ssd_step_ex(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                float* state, int batch, int nheads, int headdim, int ngroups, int dstate,
                const ssd_input_options* options, void* y, cudaStream_t stream) {
    if (!x || !dt || !A || !B || !C || !state || !y) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0) return SSD_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (headdim != 64 || !supported_dstate(dstate)) return SSD_ERR_UNSUPPORTED;
    if (batch > 65535 || nheads > 2147483647 / 64) return SSD_ERR_UNSUPPORTED;
    if (!aligned16(state) || ((uintptr_t)x & 1u) || ((uintptr_t)B & 1u) || ((uintptr_t)C & 1u) ||
        ((uintptr_t)y & 1u) || ((uintptr_t)dt & 3u) || ((uintptr_t)A & 3u) || (D && ((uintptr_t)D & 3u)))
        return SSD_ERR_INVALID_ARG;
    DtOpts dto;
    OutOpts oo;
    const int r = read_options(options, D, false, &dto, &oo);
    if (r != SSD_OK) return r;
    return launch_step(static_cast<const __nv_bfloat16*>(x), dt, A, static_cast<const __nv_bfloat16*>(B),
                       static_cast<const __nv_bfloat16*>(C), oo.Dp != nullptr ? nullptr : D, state, batch, nheads,
                       ngroups, dstate, static_cast<__nv_bfloat16*>(y), stream, dto, oo);
}

int ssd_step_multi(const void* x, const float* dt, const float* A, const void* B, const void* C, const float* D,
                   float* state, int batch, int ntokens, int nheads, int headdim, int ngroups, int dstate, void* y,
                   cudaStream_t stream) {
    if (!x || !dt || !A || !B || !C || !state || !y) return SSD_ERR_INVALID_ARG;
    if (batch <= 0 || ntokens <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
        return SSD_ERR_INVALID_ARG;
    if (nheads % ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (headdim != 64 || !supported_dstate(dstate)) return SSD_ERR_UNSUPPORTED;
    if (batch > 65535 || (int64_t)batch * ntokens * nheads > ((int64_t)1 << 40)) return SSD_ERR_UNSUPPORTED;
    if (!aligned16(state) || ((uintptr_t)x & 1u) || ((uintptr_t)B & 1u) || ((uintptr_t)C & 1u) ||
        ((uintptr_t)y & 1u) || ((uintptr_t)dt & 3u) || ((uintptr_t)A & 3u) || (D && ((uintptr_t)D & 3u)))
        return SSD_ERR_INVALID_ARG;
    return launch_step_multi(static_cast<const __nv_bfloat16*>(x), dt, A, static_cast<const __nv_bfloat16*>(B),
                             static_cast<const __nv_bfloat16*>(C), D, state, batch, ntokens, nheads, ngroups, dstate,
                             static_cast<__nv_bfloat16*>(y), stream);
}

int ssd_get_device_error(void) {
    int v[2] = {0, 0};
    const int zero[2] = {0, 0};
    if (cudaMemcpyFromSymbol(v, g_ssd_device_error, sizeof(v)) != cudaSuccess) return SSD_ERR_CUDA;
    if ((v[0] != 0 || v[1] != 0) && cudaMemcpyToSymbol(g_ssd_device_error, zero, sizeof(zero)) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (v[0] != 0) return SSD_ERR_TIMEOUT;
    return v[1] != 0 ? SSD_ERR_RANGE : SSD_OK;
}

int ssd_debug_set_wait_limit_ns(unsigned long long ns) {
    g_wait_ns.store(ns == 0 ? 1000000000ull : ns);
    return SSD_OK;
}

int ssd_debug_stall(int kinds) {
    g_stall_kinds.store(kinds);
    return SSD_OK;
}

int ssd_profile_enable(int kinds) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_mask = static_cast<unsigned>(kinds);
    return SSD_OK;
}

int ssd_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& p : g_prof_open) {
        cudaEventSynchronize(p.stop);
        g_prof_free.push_back(p.start);
        g_prof_free.push_back(p.stop);
    }
    g_prof_open.clear();
    for (int k = 0; k < kNumKinds; ++k) {
        g_prof_ms[k] = 0.0;
        g_prof_count[k] = 0;
    }
    return SSD_OK;
}

int ssd_profile_read(float* total_ms, int* launches, int max_kinds, int* n_kinds) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    int status = SSD_OK;
    for (auto& p : g_prof_open) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess)
            status = SSD_ERR_CUDA;
        g_prof_ms[p.kind] += ms;
        g_prof_count[p.kind] += 1;
        g_prof_free.push_back(p.start);
        g_prof_free.push_back(p.stop);
    }
    g_prof_open.clear();
    const int n = max_kinds < kNumKinds ? max_kinds : kNumKinds;
    for (int k = 0; k < n; ++k) {
        if (total_ms) total_ms[k] = (float)g_prof_ms[k];
        if (launches) launches[k] = g_prof_count[k];
    }
    if (n_kinds) *n_kinds = kNumKinds;
    return status;
}

const char* ssd_kernel_name(int kind) {
    return (kind >= 0 && kind < kNumKinds) ? kKindNames[kind] : "unknown";
}

long long ssd_launch_count(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    return g_launches;
}

}  // extern "C"
