// C ABI of the HLA-2 library: argument checks, segmentation plan, kernel dispatch.
// The declarations and their documentation are in include/hla2.h.
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <stdlib.h>
#include <string.h>

#include <functional>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"

namespace hla2 {
int launch_fwd_chunk_mma_d16(const ChunkArgs&, int, int, bool, cudaStream_t);
int launch_fwd_chunk_mma_d32(const ChunkArgs&, int, int, bool, cudaStream_t);
int launch_fwd_chunk_mma_d64(const ChunkArgs&, int, int, bool, cudaStream_t);
int launch_fwd_chunk_mma_d128(const ChunkArgs&, int, int, bool, cudaStream_t);
size_t fwd_chunk_mma_smem_d16(int, bool);
size_t fwd_chunk_mma_smem_d32(int, bool);
size_t fwd_chunk_mma_smem_d64(int, bool);
size_t fwd_chunk_mma_smem_d128(int, bool);

int launch_fwd_chunk_mma(const ChunkArgs& a, int d, int dv, int W, int mode, bool cm,
                         cudaStream_t st) {
    if (d != dv) return -2;
    switch (d) {
        case 16: return launch_fwd_chunk_mma_d16(a, W, mode, cm, st);
        case 32: return launch_fwd_chunk_mma_d32(a, W, mode, cm, st);
        case 64: return launch_fwd_chunk_mma_d64(a, W, mode, cm, st);
        case 128: return launch_fwd_chunk_mma_d128(a, W, mode, cm, st);
        default: return -2;
    }
}

int launch_bwd_chunk_mma_d16(const BwdArgs&, int, bool, cudaStream_t);
int launch_bwd_chunk_mma_d32(const BwdArgs&, int, bool, cudaStream_t);
int launch_bwd_chunk_mma_d64(const BwdArgs&, int, bool, cudaStream_t);
int launch_bwd_chunk_mma_d128(const BwdArgs&, int, bool, cudaStream_t);
size_t bwd_chunk_mma_smem_d16(int);
size_t bwd_chunk_mma_smem_d32(int);
size_t bwd_chunk_mma_smem_d64(int);
size_t bwd_chunk_mma_smem_d128(int);

int launch_bwd_chunk_mma(const BwdArgs& a, int d, int W, bool rsum, cudaStream_t st) {
    switch (d) {
        case 16: return launch_bwd_chunk_mma_d16(a, W, rsum, st);
        case 32: return launch_bwd_chunk_mma_d32(a, W, rsum, st);
        case 64: return launch_bwd_chunk_mma_d64(a, W, rsum, st);
        case 128: return launch_bwd_chunk_mma_d128(a, W, rsum, st);
        default: return -2;
    }
}

size_t bwd_chunk_mma_smem(int d, int W) {
    switch (d) {
        case 16: return bwd_chunk_mma_smem_d16(W);
        case 32: return bwd_chunk_mma_smem_d32(W);
        case 64: return bwd_chunk_mma_smem_d64(W);
        case 128: return bwd_chunk_mma_smem_d128(W);
        default: return 0;
    }
}

size_t fwd_chunk_mma_smem(int d, int dv, int W, bool cm) {
    if (d != dv) return 0;
    switch (d) {
        case 16: return fwd_chunk_mma_smem_d16(W, cm);
        case 32: return fwd_chunk_mma_smem_d32(W, cm);
        case 64: return fwd_chunk_mma_smem_d64(W, cm);
        case 128: return fwd_chunk_mma_smem_d128(W, cm);
        default: return 0;
    }
}
}  // namespace hla2

using namespace hla2;

namespace {

thread_local std::string g_last_error;

// NVTX ranges for profilers (a no-op unless a tool is attached): one range per C-ABI call,
// and inside the chunked forwards one range per phase (carry-in, segment summaries,
// inter-segment scan, output pass, final state).
struct NvtxScope {
    int depth = 0;
    explicit NvtxScope(const char* name) { push(name); }
    NvtxScope(const NvtxScope&) = delete;
    NvtxScope& operator=(const NvtxScope&) = delete;
    void push(const char* name) {
        nvtxRangePushA(name);
        ++depth;
    }
    void pop() {
        if (depth > 0) {
            nvtxRangePop();
            --depth;
        }
    }
    void phase(const char* name) {  // replace the current phase range
        if (depth > 1) pop();
        if (name) push(name);
    }
    ~NvtxScope() {
        while (depth > 0) pop();
    }
};
const char* const kPhaseNames[6] = {"carry-in", "segment summaries", "inter-segment scan", "output pass",
                                    "final state", nullptr};

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int succeed() {
    g_last_error.clear();
    return HLA2_OK;
}

}  // namespace

namespace hla2 {
// Records the message returned by hla2_last_error() for entry points in other files.
int set_last_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}
}  // namespace hla2

namespace {

int cuda_fail(const char* what) {
    const cudaError_t e = cudaGetLastError();
    return fail(HLA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool dim_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

struct DevInfo {
    int sms = 152;                  // GB300 when no device can be queried
    int smem_optin = 232448;        // 227 KB per block
    int smem_per_sm = 233472;       // 228 KB per SM
    int smem_reserved = 1024;       // per block
};

DevInfo dev_info() {
    DevInfo di;
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return di;
    }
    auto get = [&](cudaDeviceAttr attr, int* dst) {
        if (cudaDeviceGetAttribute(&v, attr, dev) == cudaSuccess)
            *dst = v;
        else
            cudaGetLastError();
    };
    get(cudaDevAttrMultiProcessorCount, &di.sms);
    get(cudaDevAttrMaxSharedMemoryPerBlockOptin, &di.smem_optin);
    get(cudaDevAttrMaxSharedMemoryPerMultiprocessor, &di.smem_per_sm);
    get(cudaDevAttrReservedSharedMemoryPerBlock, &di.smem_reserved);
    return di;
}

// CTAs of a chunk kernel resident on one SM, from its shared memory and thread count
// (the kernels' register budgets allow at least this many), at most `cap`.
int blocks_per_sm(size_t smem, int threads, int cap, const DevInfo& di) {
    long b = (long)di.smem_per_sm / (long)(smem + (size_t)di.smem_reserved);
    b = b < 2048 / threads ? b : 2048 / threads;
    b = b < cap ? b : cap;
    return b < 1 ? 1 : (int)b;
}

// Cut each head's chunks into segments.  The chunk passes run one CTA per segment and
// process a segment's chunks one after another, so a pass takes about
// waves x chunks-per-segment chunk steps, with waves = ceil(segments / resident CTAs).
// The segment count per head minimises that (plus a small charge per segment for the
// inter-segment scan), for `per_sm` resident CTAs per SM.
// The same cut for a call whose passes run at two residencies: passes of weight wa at per_sm_a
// resident CTAs and passes of weight wb at per_sm_b, cost = sum of weight x waves x chunks.
Plan make_plan2(int B, int H, int n, int d, int dv, int W, int sms, int per_sm_a, double wa, int per_sm_b,
                double wb);

Plan make_plan(int B, int H, int n, int d, int dv, int W, int sms, int per_sm) {
    return make_plan2(B, H, n, d, dv, W, sms, per_sm, 1.0, per_sm, 0.0);
}

Plan make_plan2(int B, int H, int n, int d, int dv, int W, int sms, int per_sm_a, double wa, int per_sm_b,
                double wb) {
    Plan p;
    p.BH = B * H;
    p.H = H;
    p.n = n;
    p.d = d;
    p.dv = dv;
    p.W = W;
    p.nchunks = (n + W - 1) / W;
    if (p.nchunks == 0 || p.BH == 0) {
        p.seg_chunks = 1;
        p.nseg = 0;
        return p;
    }
    const long sm = sms < 1 ? 1 : sms;
    const long slots_a = (long)(per_sm_a < 1 ? 1 : per_sm_a) * sm, slots_b = (long)(per_sm_b < 1 ? 1 : per_sm_b) * sm;
    const long slots = slots_a > slots_b ? slots_a : slots_b;
    long max_ph = (4 * slots + p.BH - 1) / p.BH;
    if (max_ph < 1) max_ph = 1;
    if (max_ph > p.nchunks) max_ph = p.nchunks;
    long best_sc = p.nchunks;
    double best = -1.0;
    for (long ph = 1; ph <= max_ph; ++ph) {
        const long sc = (p.nchunks + ph - 1) / ph;
        const long ns = (p.nchunks + sc - 1) / sc;
        const long waves_a = ((long)p.BH * ns + slots_a - 1) / slots_a;
        const long waves_b = ((long)p.BH * ns + slots_b - 1) / slots_b;
        const double cost = (wa * (double)waves_a + wb * (double)waves_b) * (double)sc + 0.05 * (double)ns;
        if (best < 0.0 || cost < best - 1e-9) {
            best = cost;
            best_sc = sc;
        }
    }
    p.seg_chunks = (int)best_sc;
    p.nseg = (p.nchunks + p.seg_chunks - 1) / p.seg_chunks;
    return p;
}

enum class Path { kTc, kMma, kSimt, kNone };

// HLA2_KERNEL=mma forces the mma.sync chunk kernel where the tcgen05 one would be chosen
// (used to test both paths on the same inputs).
bool tc_disabled() {
    const char* e = getenv("HLA2_KERNEL");
    return e && strcmp(e, "mma") == 0;
}

Path choose_forward_path(int dtype, int d, int dv, int W, int normalize, bool want_final, const DevInfo& di,
                         bool unmasked = false) {
    (void)want_final;  // the tcgen05 kernels have both outputs, with or without the final state,
                       // and the masked one also ratio-normalised
    if (dtype == HLA2_BF16 && d == 64 && dv == 64 && W == 128 && !(normalize && unmasked) && !tc_disabled() &&
        fwd_chunk_tc_smem() <= (size_t)di.smem_optin && fwd_chunk_tc_available())
        return Path::kTc;
    if (dtype == HLA2_BF16) {
        const size_t s = fwd_chunk_mma_smem(d, dv, W, true);
        if (s > 0 && s <= (size_t)di.smem_optin) return Path::kMma;
    }
    if (fwd_chunk_simt_smem(d, dv, W, true) <= (size_t)di.smem_optin) return Path::kSimt;
    return Path::kNone;
}

int mma_threads(int d) { return 32 * (d <= 32 ? 4 : (d == 64 ? 8 : 16)); }

// Resident CTAs per SM of the forward chunk kernels on `path`.
int forward_per_sm(Path path, int d, int dv, int W, const DevInfo& di) {
    switch (path) {
        case Path::kTc: return blocks_per_sm(fwd_chunk_tc_smem(), 288, 2, di);
        case Path::kMma: return blocks_per_sm(fwd_chunk_mma_smem(d, dv, W, false), mma_threads(d), 4, di);
        case Path::kSimt: return blocks_per_sm(fwd_chunk_simt_smem(d, dv, W, false), 256, kSimtFwdCtas, di);
        default: return 2;
    }
}

Plan forward_plan(int B, int H, int n, int d, int dv, int W, int dtype, int normalize, bool want_final,
                  const DevInfo& di) {
    const Path path = choose_forward_path(dtype, d, dv, W, normalize, want_final, di);
    return make_plan(B, H, n, d, dv, W, di.sms, forward_per_sm(path, d, dv, W, di));
}

// Chunk width a forward call runs at: the widest one <= chunk with a forward kernel for these
// sizes (the output does not depend on the width, only the rounding order does); 0 if none.
int forward_width(int dtype, int d, int dv, int chunk, int normalize, const DevInfo& di) {
    for (int W = chunk; W >= 16; W /= 2)
        if (choose_forward_path(dtype, d, dv, W, normalize, false, di) != Path::kNone) return W;
    return 0;
}

int check_common(int B, int H, int n, int d, int dv, int dtype, int normalize) {
    if (B < 0 || H < 0 || n < 0) return fail(HLA2_ERR_INVALID_ARG, "B, H, n must be >= 0 (got %d, %d, %d)", B, H, n);
    if ((long)B * H > (1L << 30)) return fail(HLA2_ERR_INVALID_ARG, "B*H too large");
    if (!dim_ok(d) || !dim_ok(dv))
        return fail(HLA2_ERR_INVALID_ARG, "d and dv must be 16, 32, 64 or 128 (got %d, %d)", d, dv);
    if (dtype != HLA2_F32 && dtype != HLA2_BF16) return fail(HLA2_ERR_INVALID_ARG, "dtype must be HLA2_F32 or HLA2_BF16");
    if (normalize != 0 && normalize != 1) return fail(HLA2_ERR_INVALID_ARG, "normalize must be 0 or 1");
    return HLA2_OK;
}

// Summaries kept per head: nseg - 1, or nseg with a final state (the tcgen05 path keeps the last
// segment's summary for the final combine; the other paths use a part of that space).
int forward_nsum(const Plan& p, bool want_final) { return want_final ? p.nseg : p.nseg - 1; }

size_t forward_ws(const Plan& p, bool want_final) {
    return p.nseg > 0 ? fwd_layout(p, forward_nsum(p, want_final)).total * sizeof(float) : 0;
}

}  // namespace

namespace {
int forward_saving_for_backward(const void* q, const void* k, const void* v, void* out, int B, int H, int n, int d,
                                int dv, const float* gamma, int normalize, int chunk, cudaStream_t st,
                                const hla2_opts* opts);
// Plain forward on the tcgen05 first-order scans (bf16, d = dv = 128, chunk >= 128, masked,
// unnormalised, no state in or out): its workspace bytes (0: not this path), and the call.
size_t fo_forward_ws(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize, bool want_final);
int fo_forward_call(const void* q, const void* k, const void* v, void* out, int B, int H, int n, const float* gamma,
                    cudaStream_t st, const hla2_opts* opts);
Plan fo_plan(int B, int H, int n, int d, const DevInfo& di);
}  // namespace

extern "C" {

int hla2_version(void) { return 100; }

const char* hla2_last_error(void) { return g_last_error.c_str(); }

size_t hla2_state_floats(int d, int dv) { return raw_state_floats(d, dv); }

size_t hla2_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                    int normalize, int want_final_state) {
    if (check_common(B, H, n, d, dv, dtype, normalize) != HLA2_OK || !dim_ok(chunk)) return (size_t)-1;
    const DevInfo di = dev_info();
    const int W = forward_width(dtype, d, dv, chunk, normalize, di);
    if (!W) return (size_t)-1;  // hla2_forward rejects these sizes (HLA2_ERR_UNSUPPORTED)
    const size_t ws = forward_ws(forward_plan(B, H, n, d, dv, W, dtype, normalize, want_final_state != 0, di),
                                 want_final_state != 0);
    // masked calls without init_state run on the first-order scans; the unmasked output and
    // calls with init_state keep the chunk kernels (what the query does not see): the larger
    const size_t fo = fo_forward_ws(B, H, n, d, dv, chunk, dtype, normalize, want_final_state != 0);
    return fo > ws ? fo : ws;
}

int hla2_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n,
                 int d, int dv, const float* gamma, int normalize, int chunk, hla2_stream_t stream,
                 const hla2_opts* opts) {
    NvtxScope nvtx("hla2_forward");
    if (!opts) return fail(HLA2_ERR_INVALID_ARG, "opts must not be NULL");
    int rc = check_common(B, H, n, d, dv, opts->dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    if (normalize && !isfinite(opts->eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (opts->flags & ~(HLA2_FLAG_SAVE_FOR_BACKWARD | HLA2_FLAG_UNMASKED))
        return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_forward");
    const bool unmasked = (opts->flags & HLA2_FLAG_UNMASKED) != 0;
    if (unmasked && (opts->flags & HLA2_FLAG_SAVE_FOR_BACKWARD))
        return fail(HLA2_ERR_UNSUPPORTED, "the backward covers the masked output only");
    const long BH = (long)B * H;
    const bool want_final = opts->final_state != nullptr;
    if ((opts->init_state && !aligned16(opts->init_state)) || (want_final && !aligned16(opts->final_state)))
        return fail(HLA2_ERR_INVALID_ARG, "init_state / final_state must be 16-byte aligned");
    if (BH == 0) return succeed();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t sf = raw_state_floats(d, dv);
    if (n == 0) {
        // no tokens: the final state is the initial one (or the empty prefix); the unmasked
        // variant reports G = h = 0 as for any other length
        if (want_final) {
            cudaError_t e = opts->init_state
                                ? cudaMemcpyAsync(opts->final_state, opts->init_state, BH * sf * sizeof(float),
                                                  cudaMemcpyDeviceToDevice, st)
                                : cudaMemsetAsync(opts->final_state, 0, BH * sf * sizeof(float), st);
            if (e == cudaSuccess && unmasked && opts->init_state) {
                const PackOff po = pack_off(d, dv);
                e = cudaMemset2DAsync(opts->final_state + po.G, sf * sizeof(float), 0, (size_t)d * dv * sizeof(float),
                                      (size_t)BH, st);
                if (e == cudaSuccess)
                    e = cudaMemset2DAsync(opts->final_state + po.h, sf * sizeof(float), 0, (size_t)d * sizeof(float),
                                          (size_t)BH, st);
            }
            if (e != cudaSuccess) return cuda_fail("final state copy");
        }
        return succeed();
    }
    if (!q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must not be NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
    {
        // out is written while q, k, v are still being read (and, on the stored-p path, holds
        // the summary pass's p until the output pass replaces it)
        const size_t es = opts->dtype == HLA2_BF16 ? 2 : 4;
        const size_t rows = (size_t)BH * (size_t)n, nq = rows * d * es, nv = rows * dv * es;
        if (overlaps(out, nv, q, nq) || overlaps(out, nv, k, nq) || overlaps(out, nv, v, nv))
            return fail(HLA2_ERR_INVALID_ARG, "out must not overlap q, k or v");
    }
    if (opts->flags & HLA2_FLAG_SAVE_FOR_BACKWARD)
        return forward_saving_for_backward(q, k, v, out, B, H, n, d, dv, gamma, normalize, chunk, st, opts);

    const DevInfo di = dev_info();
    if (!unmasked && !opts->init_state && fo_forward_ws(B, H, n, d, dv, chunk, opts->dtype, normalize, want_final))
        return fo_forward_call(q, k, v, out, B, H, n, gamma, st, opts);  // (at the width asked for)
    {
        const int W = forward_width(opts->dtype, d, dv, chunk, normalize, di);
        if (!W) return fail(HLA2_ERR_UNSUPPORTED, "no kernel for dtype %d, d %d, dv %d, chunk %d", opts->dtype, d, dv, chunk);
        chunk = W;  // everything below runs at the width the kernels cover
    }
    const Path path = choose_forward_path(opts->dtype, d, dv, chunk, normalize, want_final, di, unmasked);
    // The unmasked output keeps the masked call's segmentation, so the workspace query
    // (which has no flags) covers it: it uses a subset of the masked workspace.
    const Plan p = unmasked ? forward_plan(B, H, n, d, dv, chunk, opts->dtype, normalize, want_final, di)
                            : make_plan(B, H, n, d, dv, chunk, di.sms, forward_per_sm(path, d, dv, chunk, di));
    const FwdLayout L = fwd_layout(p, forward_nsum(p, want_final));
    const size_t need = L.total * sizeof(float);
    if (!opts->workspace || opts->workspace_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    // tcgen05 path with a final state (masked): every segment's summary is kept, and the last
    // one is combined with the carry into the last segment after the output pass
    const bool tc_final = path == Path::kTc && want_final;

    ChunkArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.BH = (int)BH;
    a.H = H;
    a.n = n;
    a.W = chunk;
    a.nchunks = p.nchunks;
    a.seg_chunks = p.seg_chunks;
    a.nseg = p.nseg;
    a.nsum = tc_final ? p.nseg : p.nseg - 1;
    a.gamma = gamma;
    a.normalize = normalize;
    a.eps = opts->eps;
    a.want_final = want_final ? 1 : 0;
    a.ws = static_cast<float*>(opts->workspace);
    a.L = L;
    a.unmasked = unmasked ? 1 : 0;

    const bool bf = opts->dtype == HLA2_BF16;
    // tcgen05 path with more than one segment (or a final state, or normalised): the summary
    // pass also stores the segment-local p_t = S_t q_t in out, over every segment, and the
    // output pass starts from it (kOutputP), so that only Z (unmasked: C) is carried from chunk
    // to chunk there.  Its q and p moments per segment (the y carry of the denominator and of
    // the final state) come from the moments kernel.
    const bool stored_p = path == Path::kTc && (p.nseg > 1 || tc_final || normalize);
    // (the masked summary pass forms them itself; the unmasked final state runs the kernel)
    const bool tc_moments = path == Path::kTc && unmasked && tc_final;
    auto chunk_pass = [&](int seg0, int count, bool summary, bool cm) -> int {
        ChunkArgs b = a;
        b.seg0 = seg0;
        b.nseg_launch = count;
        if (path == Path::kTc)
            return launch_fwd_chunk_tc(b, summary ? (stored_p ? kSummaryP : kSummary) : (stored_p ? kOutputP : kOutput),
                                       reinterpret_cast<int*>(a.ws), st);
        if (path == Path::kMma) return launch_fwd_chunk_mma(b, d, dv, chunk, summary ? kSummary : kOutput, cm, st);
        return launch_fwd_chunk_simt(b, d, dv, chunk, summary, cm, bf, st);
    };

    auto mark = [&](int i) {
        nvtx.phase(kPhaseNames[i]);
        if (opts->phase_events && i < opts->n_phase_events && opts->phase_events[i] &&
            cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[i]), st) != cudaSuccess)
            cudaGetLastError();  // a bad profiling handle must not fail the computation
    };
    cudaGetLastError();  // launch errors below are ours
    mark(0);
    if (launch_init_carry(a, d, dv, opts->init_state, st)) return cuda_fail("carry-in initialisation");
    mark(1);
    if (stored_p && p.nseg == 1) {  // one segment: its p (a final state: its summary and moments)
        if (chunk_pass(0, 1, true, true)) return cuda_fail("segment summaries");
        if (tc_moments && launch_seg_moments64(a, st)) return cuda_fail("segment moments");
        mark(2);
    } else if (p.nseg > 1) {
        const int steps = p.nseg - 1, seg_tokens = p.seg_chunks * chunk;
        const size_t dd = (size_t)d * d, ddv = (size_t)d * dv;
        if (chunk_pass(0, stored_p ? p.nseg : steps, true, true)) return cuda_fail("segment summaries");
        if (tc_moments && launch_seg_moments64(a, st)) return cuda_fail("segment moments");
        mark(2);
        // independent decayed prefixes share a launch (one alone keeps the plain scan kernel)
        auto scans = [&](const ScanJob* jobs, int njobs) {
            if (njobs == 1)
                return launch_linear_scan(jobs[0].src, jobs[0].dst, a.BH, H, steps, jobs[0].E, jobs[0].src_hs,
                                          jobs[0].dst_hs, jobs[0].store_all != 0, gamma, seg_tokens, jobs[0].power,
                                          st);
            return launch_linear_scans(jobs, njobs, a.BH, H, steps, gamma, seg_tokens, st);
        };
        const size_t dsz = (size_t)d;
        ScanJob first[kMaxScanJobs];
        int nfirst = 0;
        first[nfirst++] = {a.ws + L.SB, a.ws + L.Sin, dd, a.nsum * dd, p.nseg * dd, 1, 1};
        if (unmasked) {
            // unmasked monoid: C and m (in the Z and y slots) are plain decayed prefixes
            first[nfirst++] = {a.ws + L.ZB, a.ws + L.Zin, ddv, a.nsum * ddv, p.nseg * ddv, 1, 1};
            if (normalize || want_final) first[nfirst++] = {a.ws + L.yB, a.ws + L.yin, dsz, a.nsum * dsz, p.nseg * dsz, 1, 1};
        } else if (want_final) {  // C and m carried into the last segment
            first[nfirst++] = {a.ws + L.CB, a.ws + L.Clast, ddv, a.nsum * ddv, ddv, 0, 1};
            first[nfirst++] = {a.ws + L.mB, a.ws + L.mlast, dsz, a.nsum * dsz, dsz, 0, 1};
        }
        if (scans(first, nfirst)) return cuda_fail("key-moment scan");
        // the denominator moment y is read only by the normalised output and the final state
        const bool with_y = normalize || want_final;
        if (!unmasked) {
            if (launch_cross(a, d, dv, with_y, st)) return cuda_fail("cross terms");
            const ScanJob second[2] = {{a.ws + L.ZB, a.ws + L.Zin, ddv, a.nsum * ddv, p.nseg * ddv, 1, 2},
                                       {a.ws + L.yB, a.ws + L.yin, dsz, a.nsum * dsz, p.nseg * dsz, 1, 2}};
            if (scans(second, with_y ? 2 : 1)) return cuda_fail("masked-summary scan");
        }
    } else {
        mark(2);
    }
    mark(3);
    if (want_final && p.nseg > 1 && !unmasked && !tc_final) {
        if (chunk_pass(0, p.nseg - 1, false, false) || chunk_pass(p.nseg - 1, 1, false, true))
            return cuda_fail("output pass");
    } else {
        if (chunk_pass(0, p.nseg, false, want_final)) return cuda_fail("output pass");
    }
    mark(4);
    if (tc_final) {
        if (launch_final_combine64(a, opts->final_state, st)) return cuda_fail("final state");
    } else if (want_final && launch_finalize(a, d, dv, opts->final_state, st)) {
        return cuda_fail("final state");
    }
    mark(5);
    return succeed();
}

int hla2_workspace_status(const void* workspace, hla2_stream_t stream) {
    if (!workspace) return fail(HLA2_ERR_INVALID_ARG, "workspace must not be NULL");
    int code = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&code, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return cuda_fail("status read");
    if (code != 0) return fail(HLA2_ERR_TIMEOUT, "a bounded device-side wait gave up (site %d)", code);
    return succeed();
}

int hla2_debug_status(int clear) {
#ifdef HLA2_DEBUG
    int (*const readers[])(bool) = {dbg_read_fwd_simt,    dbg_read_decode,      dbg_read_fwd_mma_d16,
                                    dbg_read_fwd_mma_d32, dbg_read_fwd_mma_d64, dbg_read_fwd_mma_d128,
                                    dbg_read_bwd_mma_d16, dbg_read_bwd_mma_d32, dbg_read_bwd_mma_d64,
                                    dbg_read_bwd_mma_d128, dbg_read_bwd_simt,   dbg_read_scan,
                                    dbg_read_fo_tc,       dbg_read_fo64_tc,     dbg_read_selftest};
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail("debug status");
    int site = 0;
    for (auto rd : readers) {
        const int v = rd(clear != 0);
        if (v < 0) return cuda_fail("debug status read");
        if (!site) site = v;
    }
    succeed();
    return site;
#else
    (void)clear;
    return fail(HLA2_ERR_UNSUPPORTED, "not a debug build (compile with HLA2_DEBUG)");
#endif
}

int hla2_debug_selftest(hla2_stream_t stream) {
#ifdef HLA2_DEBUG
    cudaGetLastError();
    if (launch_debug_check_selftest(reinterpret_cast<cudaStream_t>(stream))) return cuda_fail("debug self-test");
    return succeed();
#else
    (void)stream;
    return fail(HLA2_ERR_UNSUPPORTED, "not a debug build (compile with HLA2_DEBUG)");
#endif
}

int hla2_selftest_wait_timeout(void* workspace, hla2_stream_t stream) {
    if (!workspace || !aligned16(workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    cudaGetLastError();
    if (launch_wait_timeout_selftest(static_cast<int*>(workspace), reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("wait self-test");
    return succeed();
}

int hla2_forward_plan(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize,
                      int want_final_state, int* nseg, int* seg_chunks, int* launches) {
    int rc = check_common(B, H, n, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    const DevInfo di = dev_info();
    const int W = forward_width(dtype, d, dv, chunk, normalize, di);
    if (!W) return fail(HLA2_ERR_UNSUPPORTED, "no forward kernel for d %d, dv %d at chunk <= %d", d, dv, chunk);
    if (fo_forward_ws(B, H, n, d, dv, chunk, dtype, normalize, want_final_state != 0)) {
        // first-order scans: S summaries, zero (+ scan), p pass, (p, v) summaries (with a final
        // state: the pass that also forms the (q, v) summaries and the moments), zero (+ scan),
        // output pass; with a final state also the final combine (+ the last-only scans of C, m, y)
        const Plan p = fo_plan(B, H, n, d, di);
        const bool many = p.nseg > 1;
        if (nseg) *nseg = p.nseg;
        if (seg_chunks) *seg_chunks = p.seg_chunks;
        if (launches)
            *launches = p.nseg > 0 ? 6 + (many ? 2 : 0) + (want_final_state ? 1 + (many ? 1 : 0) : 0) : 0;
        return succeed();
    }
    chunk = W;
    const Plan p = forward_plan(B, H, n, d, dv, chunk, dtype, normalize, want_final_state != 0, di);
    int l = 0;
    const bool tc = choose_forward_path(dtype, d, dv, chunk, normalize, want_final_state != 0, di) == Path::kTc;
    // (the launch counts of the masked output; independent scans share one launch: S with C
    // and m, Z with y)
    if (p.nseg > 0 && want_final_state && tc) {
        // carry-in, summary (with the segment moments), output, final combine; the S (C, m)
        // scan, cross terms, the Z (y) scan
        l = 4 + (p.nseg > 1 ? 3 : 0);
    } else if (p.nseg > 0 && normalize && tc) {
        // carry-in, summary (it stores p and forms the moments), output; S scan, cross terms,
        // the Z (y) scan
        l = 3 + (p.nseg > 1 ? 3 : 0);
    } else if (p.nseg > 0) {
        l = 2;                                                   // carry-in, output pass
        if (p.nseg > 1) l += 4;                                  // summary, S (C, m) scan, cross, Z (y) scan
        if (want_final_state) l += 1 + (p.nseg > 1 ? 1 : 0);     // finalize, last-segment pass
    } else if (want_final_state && (long)B * H > 0) {
        l = 0;                                                   // a copy or memset only
    }
    if (nseg) *nseg = p.nseg;
    if (seg_chunks) *seg_chunks = p.seg_chunks;
    if (launches) *launches = l;
    return succeed();
}

}  // extern "C"

namespace {

// The backward runs its chunk passes at the largest width <= chunk whose kernels are
// compiled and fit in shared memory (the result does not depend on the width).
int backward_width(int d, int chunk, const DevInfo& di) {
    for (int W = chunk; W >= 16; W /= 2) {
        const size_t sb = bwd_chunk_mma_smem(d, W), sf = fwd_chunk_mma_smem(d, d, W, true);
        if (sb > 0 && sf > 0 && sb <= (size_t)di.smem_optin && sf <= (size_t)di.smem_optin) return W;
    }
    return 0;
}

// Resident CTAs per SM of the backward's chunk passes (the forward passes at width W and
// the reverse-mode passes run with the same segmentation).
int backward_per_sm(int d, int W, const DevInfo& di) {
    const int b = blocks_per_sm(bwd_chunk_mma_smem(d, W), mma_threads(d), 4, di);
    const int f = blocks_per_sm(fwd_chunk_mma_smem(d, d, W, false), mma_threads(d), 4, di);
    return b < f ? b : f;
}

struct BwdLayout {
    FwdLayout F;              // forward pieces (nseg summaries)
    size_t states_bytes_off;  // byte offset of the bf16 chunk states
    size_t ZhB, ShB, Zh_end, Sh_end;  // float offsets
    size_t total_bytes;
};

BwdLayout bwd_layout(const Plan& p, size_t state_elem = sizeof(bf16)) {
    BwdLayout L;
    L.F = fwd_layout(p, p.nseg);
    const size_t BH = p.BH, ns = p.nseg, dd = (size_t)p.d * p.d, ddv = (size_t)p.d * p.dv;
    size_t o = L.F.total;
    L.ZhB = o;    o = align64(o + BH * ns * ddv);
    L.ShB = o;    o = align64(o + BH * ns * dd);
    L.Zh_end = o; o = align64(o + BH * ns * ddv);
    L.Sh_end = o; o = align64(o + BH * ns * dd);
    L.states_bytes_off = o * sizeof(float);
    L.total_bytes = L.states_bytes_off + BH * (size_t)p.nchunks * (dd + ddv) * state_elem;
    return L;
}

// The fp32 backward (SIMT kernels) runs at the largest width <= min(chunk, 32) whose forward
// and reverse kernels fit in shared memory.
int backward_width_f32(int d, int dv, int chunk, const DevInfo& di) {
    for (int W = chunk < 32 ? chunk : 32; W >= 16; W /= 2)
        if (bwd_chunk_simt_smem(d, dv, W) <= (size_t)di.smem_optin &&
            fwd_chunk_simt_smem(d, dv, W, true) <= (size_t)di.smem_optin)
            return W;
    return 0;
}

// Width, segmentation and workspace of an unnormalised backward call (W = 0: no kernel).
struct BwdPlan {
    int W = 0;
    bool f32 = false;
    Plan p;
    BwdLayout L;
};

BwdPlan backward_plan(int B, int H, int n, int d, int dv, int chunk, int dtype, const DevInfo& di) {
    BwdPlan bp;
    bp.f32 = dtype == HLA2_F32;
    bp.W = bp.f32 ? backward_width_f32(d, dv, chunk, di) : backward_width(d, chunk, di);
    if (!bp.W) return bp;
    if (bp.f32) {
        // the two forward passes (segment summaries, state export) run at the forward kernel's
        // residency, the two reverse passes at the reverse kernel's; per chunk the reverse pair
        // costs about 1.5 times the forward pair (36 and 54 us at d = 64, dv = 80, W = 32)
        const int f = blocks_per_sm(fwd_chunk_simt_smem(d, dv, bp.W, false), 256, kSimtFwdCtas, di);
        const int b = blocks_per_sm(bwd_chunk_simt_smem(d, dv, bp.W), 256, kSimtBwdCtas, di);
        bp.p = make_plan2(B, H, n, d, dv, bp.W, di.sms, f, 1.0, b, 1.5);
    } else {
        bp.p = make_plan(B, H, n, d, dv, bp.W, di.sms, backward_per_sm(d, bp.W, di));
    }
    bp.L = bwd_layout(bp.p, bp.f32 ? sizeof(float) : sizeof(bf16));
    return bp;
}

// Chunk-pass arguments at the backward's width and segmentation.
ChunkArgs backward_chunk_args(const void* q, const void* k, const void* v, void* out, long BH, int H, int n,
                              const Plan& p, const float* gamma, void* workspace, const BwdLayout& L) {
    ChunkArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.BH = (int)BH;
    a.H = H;
    a.n = n;
    a.W = p.W;
    a.nchunks = p.nchunks;
    a.seg_chunks = p.seg_chunks;
    a.nseg = p.nseg;
    a.nsum = p.nseg;
    a.gamma = gamma;
    a.ws = static_cast<float*>(workspace);
    a.L = L.F;
    a.chunk_states = reinterpret_cast<bf16*>(static_cast<char*>(workspace) + L.states_bytes_off);
    return a;
}

// The forward pieces the reverse-mode passes consume, at the backward's width: carries at
// the segment starts (summaries of every segment, whose C_B the reverse cross term also
// reads, and the inter-segment scan), then one chunk pass that exports the bf16 (S, Z) at
// every chunk start (last_mode kStates) and also writes the output (kOutStates).
int backward_forward_part(const ChunkArgs& a, const Plan& p, const BwdLayout& L, int d, int dv, int last_mode,
                          cudaStream_t st, const std::function<void(int)>* mark) {
    float* ws = a.ws;
    const size_t dd = (size_t)d * d, ddv = (size_t)d * dv;
    const int seg_tokens = p.seg_chunks * p.W;
    auto pass = [&](int mode) {
        ChunkArgs c = a;
        c.seg0 = 0;
        c.nseg_launch = p.nseg;
        return launch_fwd_chunk_mma(c, d, dv, p.W, mode, false, st);
    };
    auto tick = [&](int i) {
        if (mark) (*mark)(i);
    };
    if (launch_init_carry(a, d, dv, nullptr, st)) return cuda_fail("carry-in initialisation");
    tick(1);
    if (p.nseg > 1) {
        const int steps = p.nseg - 1;
        if (pass(kSummary)) return cuda_fail("segment summaries");
        tick(2);
        if (launch_linear_scan(ws + L.F.SB, ws + L.F.Sin, a.BH, a.H, steps, dd, a.nsum * dd, p.nseg * dd, true,
                               a.gamma, seg_tokens, 1, st) ||
            launch_cross(a, d, dv, false, st) ||
            launch_linear_scan(ws + L.F.ZB, ws + L.F.Zin, a.BH, a.H, steps, ddv, a.nsum * ddv, p.nseg * ddv, true,
                               a.gamma, seg_tokens, 2, st))
            return cuda_fail("forward segment scan");
    } else {
        tick(2);
    }
    tick(3);
    if (pass(last_mode)) return cuda_fail(last_mode == kOutStates ? "output pass" : "forward state export");
    tick(4);
    return HLA2_OK;
}

// The same forward pieces for the fp32 backward, on the SIMT kernel: segment summaries, the
// inter-segment scan, then a pass that exports the fp32 (S, Z) at every chunk start (and, with
// out, also writes the unnormalised output there).
int backward_forward_part_f32(const ChunkArgs& a, const Plan& p, const BwdLayout& L, int d, int dv, cudaStream_t st,
                              float* out = nullptr) {
    float* ws = a.ws;
    const size_t dd = (size_t)d * d, ddv = (size_t)d * dv;
    const int seg_tokens = p.seg_chunks * p.W;
    ChunkArgs c = a;
    c.seg0 = 0;
    c.nseg_launch = p.nseg;
    if (launch_init_carry(a, d, dv, nullptr, st)) return cuda_fail("carry-in initialisation");
    if (p.nseg > 1) {
        const int steps = p.nseg - 1;
        if (launch_fwd_chunk_simt(c, d, dv, p.W, true, true, false, st)) return cuda_fail("segment summaries");
        if (launch_linear_scan(ws + L.F.SB, ws + L.F.Sin, a.BH, a.H, steps, dd, a.nsum * dd, p.nseg * dd, true,
                               a.gamma, seg_tokens, 1, st) ||
            launch_cross(a, d, dv, false, st) ||
            launch_linear_scan(ws + L.F.ZB, ws + L.F.Zin, a.BH, a.H, steps, ddv, a.nsum * ddv, p.nseg * ddv, true,
                               a.gamma, seg_tokens, 2, st))
            return cuda_fail("forward segment scan");
    }
    c.out = out;
    c.chunk_states_f32 = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + L.states_bytes_off);
    if (launch_fwd_chunk_simt(c, d, dv, p.W, false, false, false, st)) return cuda_fail("forward state export");
    return HLA2_OK;
}

// fp32 reverse-mode passes: reverse summaries, the reverse scan with its cross term, gradients.
int backward_reverse_part_f32(const float* q, const float* k, const float* v, const float* dout, float* dq, float* dk,
                              float* dvo, int H, const Plan& p, const BwdLayout& L, const float* gamma, float* ws,
                              int d, int dv, cudaStream_t st) {
    BwdArgsF b{};
    b.q = q;
    b.k = k;
    b.v = v;
    b.dout = dout;
    b.dq = dq;
    b.dk = dk;
    b.dv = dvo;
    b.BH = p.BH;
    b.H = H;
    b.n = p.n;
    b.W = p.W;
    b.nchunks = p.nchunks;
    b.seg_chunks = p.seg_chunks;
    b.nseg = p.nseg;
    b.gamma = gamma;
    b.ws = ws;
    b.ZhB = L.ZhB;
    b.ShB = L.ShB;
    b.Zh_end = L.Zh_end;
    b.Sh_end = L.Sh_end;
    b.chunk_states = reinterpret_cast<const float*>(reinterpret_cast<const char*>(ws) + L.states_bytes_off);
    BwdArgs r{};  // what the reverse cross term reads
    r.BH = p.BH;
    r.H = H;
    r.n = p.n;
    r.W = p.W;
    r.nchunks = p.nchunks;
    r.seg_chunks = p.seg_chunks;
    r.nseg = p.nseg;
    r.gamma = gamma;
    r.ws = ws;
    r.ZhB = L.ZhB;
    r.ShB = L.ShB;
    r.Zh_end = L.Zh_end;
    r.Sh_end = L.Sh_end;
    const size_t dd = (size_t)d * d, ddv = (size_t)d * dv;
    if (launch_bwd_chunk_simt(b, d, dv, true, st)) return cuda_fail("reverse summaries");
    if (launch_reverse_scan(ws + L.ZhB, ws + L.Zh_end, p.BH, H, p.nseg, ddv, gamma, p.n, p.W, p.seg_chunks, 2, st) ||
        launch_reverse_cross(r, ws + L.F.CB, d, dv, st) ||
        launch_reverse_scan(ws + L.ShB, ws + L.Sh_end, p.BH, H, p.nseg, dd, gamma, p.n, p.W, p.seg_chunks, 1, st))
        return cuda_fail("reverse segment scan");
    if (launch_bwd_chunk_simt(b, d, dv, false, st)) return cuda_fail("gradient pass");
    return HLA2_OK;
}


// ---- d = dv = 128 training path on the tcgen05 first-order scan kernel (fo_tc.cu) -----------
//
// With LA_g(x, k, v)_t = sum_{i <= t} g^(t-i) (x_t . k_i) v_i (a first-order scan; RLA_g: the
// reverse one, sum over i >= t), the masked output is two chained scans (section summary §4.2,
// technical summary item 1): p = LA_g(q, k, k) = S_t q_t and o = LA_{g^2}(q, p, v) = q_t^T Z_t.
// Its reverse mode is six more:
//   dp = RLA_{g^2}(v, dO, q)   (= Zh_t v_t,  Zh = sum q dO^T)
//   dv = RLA_{g^2}(p, q, dO)   (= Zh_t^T p_t)
//   dk = RLA_g(k, dp, q) + RLA_g(k, q, dp)   (= (Sh_t + Sh_t^T) k_t,  Sh = sum dp q^T)
//   dq = LA_{g^2}(dO, v, p) + LA_g(dp, k, k)  (= Z_t dO_t + S_t dp_t)
// Each launch runs every segment of every head with a carry from the other segments.  The
// carry of a scan whose keys are an earlier launch's output comes from summaries that launch
// forms over its own output, so every inter-segment scan is a plain decayed prefix.
// Passes: forward F1 (S summaries), F2 (p, stored, with Z summaries), F3 (o); reverse B1 (Zh
// summaries), B2 (dp, stored, with Sh summaries), B3 (dv), B4 (dk), B5a (Z dO, stored), B5b (dq).

// bf16, d == dv in {64, 128}, chunk >= 128, unnormalised, and the kernels fit this device.
bool fo_path(int dtype, int d, int dv, int chunk, int normalize, const DevInfo& di) {
    if (dtype != HLA2_BF16 || d != dv || (d != 64 && d != 128) || chunk < 128 || normalize || tc_disabled() ||
        !fo_tc_available())
        return false;
    return (d == 128 ? fo_tc_max_smem() : fo64_tc_max_smem()) <= (size_t)di.smem_optin;
}

Plan fo_plan(int B, int H, int n, int d, const DevInfo& di) { return make_plan(B, H, n, d, d, 128, di.sms, 1); }

int fo_summary(const FoArgs& a, int d, const void* k, const void* v, bool reverse, cudaStream_t st) {
    return d == 64 ? launch_fo64_tc_summary(a, k, v, reverse, st) : launch_fo_tc_summary(a, k, v, reverse, st);
}
int fo_out(const FoArgs& a, int d, const void* x, const void* k, const void* v, bool r2, int next_sum, const void* xv,
           const void* add, void* out, bool reverse, cudaStream_t st) {
    return d == 64 ? launch_fo64_tc_out(a, x, k, v, r2, next_sum, xv, add, out, reverse, st)
                   : launch_fo_tc_out(a, x, k, v, r2, next_sum, xv, add, out, reverse, st);
}

struct FoLayout {
    size_t SB, Sin, ZB, Zin, ZhB, Zhend, ShB, Shend;  // byte offsets, fp32 [BH][nseg][d][d]
    size_t P, dP, dqa;                                // byte offsets, bf16 [BH][n][d]
    // a forward with a final state (not with the backward's parts): C summaries [BH][nseg][d][d],
    // m and y moments [BH][nseg][d], the carries of C, m, y into the last segment [BH][d][d],
    // [BH][d] (contiguous, zeroed together)
    size_t CB, mB, yB, Cl, ml, yl, carries_bytes;
    size_t fwd_total, final_total, total;             // bytes kept by the forward; with a final state; by the backward
};

FoLayout fo_layout(const Plan& p) {
    FoLayout L;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t sum = (size_t)p.BH * p.nseg * p.d * p.d * sizeof(float);
    const size_t tok = (size_t)p.BH * p.n * p.d * sizeof(bf16);
    size_t o = 256;  // status word
    L.SB = o;    o = up(o + sum);
    L.Sin = o;   o = up(o + sum);
    L.ZB = o;    o = up(o + sum);
    L.Zin = o;   o = up(o + sum);
    L.P = o;     o = up(o + tok);
    L.fwd_total = o;
    {
        const size_t vec = (size_t)p.BH * p.nseg * p.d * sizeof(float);
        size_t f = o;
        L.CB = f;  f = up(f + sum);
        L.mB = f;  f = up(f + vec);
        L.yB = f;  f = up(f + vec);
        L.Cl = f;  f += (size_t)p.BH * p.d * p.d * sizeof(float);
        L.ml = f;  f += (size_t)p.BH * p.d * sizeof(float);
        L.yl = f;  f += (size_t)p.BH * p.d * sizeof(float);
        L.carries_bytes = f - L.Cl;
        L.final_total = up(f);
    }
    L.ZhB = o;   o = up(o + sum);
    L.Zhend = o; o = up(o + sum);
    L.ShB = o;   o = up(o + sum);
    L.Shend = o; o = up(o + sum);
    L.dP = o;    o = up(o + tok);
    L.dqa = o;   o = up(o + tok);
    L.total = o;
    return L;
}

FoArgs fo_args(const Plan& p, const float* gamma, char* ws) {
    FoArgs a{};
    a.BH = p.BH;
    a.H = p.H;
    a.n = p.n;
    a.nchunks = p.nchunks;
    a.seg_chunks = p.seg_chunks;
    a.nseg = p.nseg;
    a.gamma = gamma;
    a.status = reinterpret_cast<int*>(ws);
    return a;
}

// Forward scans up to the stored p: S summaries, S carries, p with the Z summaries, Z carries.
// With final_sums (d = 128, a final state asked for) the (p, v) summaries come from one pass over
// (q, p, v) that also forms the (q, v) summaries and the q and p moments the final state reads.
int fo_forward_part(const void* q, const void* k, const void* v, const Plan& p, const float* gamma, char* ws,
                    const FoLayout& L, cudaStream_t st, bool final_sums = false) {
    auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t E = (size_t)p.d * p.d;
    const int seg_tokens = p.seg_chunks * p.W;
    FoArgs a = fo_args(p, gamma, ws);
    a.pow = 1;
    a.summary = f(L.SB);
    if (fo_summary(a, p.d, k, nullptr, false, st)) return cuda_fail("key moment summaries");
    if (launch_fo_zero_first(f(L.Sin), p.BH, p.nseg, (int)E, a.status, st) ||
        (p.nseg > 1 && launch_linear_scan(f(L.SB), f(L.Sin), p.BH, p.H, p.nseg - 1, E, p.nseg * E, p.nseg * E, true,
                                          gamma, seg_tokens, 1, st)))
        return cuda_fail("key moment scan");
    // p = LA_g(q, k, k) in the pipelined order of the passes without a next summary, then the
    // (p, v) summaries at decay g^2 in a summary pass of their own
    a.pow = 1;
    a.carry = f(L.Sin);
    a.carry_mode = 0;
    if (fo_out(a, p.d, q, k, nullptr, false, 0, nullptr, nullptr, ws + L.P, false, st)) return cuda_fail("p pass");
    a.carry = nullptr;
    if (final_sums) {
        a.pow = 1;
        a.summary = f(L.CB);
        if (launch_fo_tc_summary_final(a, q, ws + L.P, v, f(L.ZB), f(L.mB), f(L.yB), st))
            return cuda_fail("final-state summaries");
    } else {
        a.pow = 2;
        a.summary = f(L.ZB);
        if (fo_summary(a, p.d, ws + L.P, v, false, st)) return cuda_fail("Z summaries");
    }
    if (launch_fo_zero_first(f(L.Zin), p.BH, p.nseg, (int)E, nullptr, st) ||
        (p.nseg > 1 && launch_linear_scan(f(L.ZB), f(L.Zin), p.BH, p.H, p.nseg - 1, E, p.nseg * E, p.nseg * E, true,
                                          gamma, seg_tokens, 2, st)))
        return cuda_fail("Z scan");
    return HLA2_OK;
}

// F3: o = LA_{g^2}(q, p, v) from the stored p and the Z carries.
int fo_output_pass(const void* q, const void* v, void* out, const Plan& p, const float* gamma, char* ws,
                   const FoLayout& L, cudaStream_t st) {
    FoArgs a = fo_args(p, gamma, ws);
    a.pow = 2;
    a.carry = reinterpret_cast<const float*>(ws + L.Zin);
    a.carry_mode = 0;
    if (fo_out(a, p.d, q, ws + L.P, v, false, 0, nullptr, nullptr, out, false, st)) return cuda_fail("output pass");
    return HLA2_OK;
}

// B1 .. B5b from the stored p and the forward carries.
int fo_reverse_part(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dvv,
                    const Plan& p, const float* gamma, char* ws, const FoLayout& L, cudaStream_t st) {
    auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t E = (size_t)p.d * p.d;
    void* P = ws + L.P;
    void* dP = ws + L.dP;
    void* dqa = ws + L.dqa;
    FoArgs a = fo_args(p, gamma, ws);
    // B1: Zh^T summaries (keys dO, values q), reverse, g^2; then the reverse scan
    a.pow = 2;
    a.summary = f(L.ZhB);
    if (fo_summary(a, p.d, dout, q, true, st)) return cuda_fail("Zh summaries");
    if (launch_reverse_scan(f(L.ZhB), f(L.Zhend), p.BH, p.H, p.nseg, E, gamma, p.n, p.W, p.seg_chunks, 2, st))
        return cuda_fail("Zh scan");
    // B2: dp = RLA_{g^2}(v, dO, q), stored; Sh summaries over (dp, q) with g
    a.pow = 2;
    a.pow_next = 1;
    a.carry = f(L.Zhend);
    a.carry_mode = 0;
    a.summary = f(L.ShB);
    if (fo_out(a, p.d, v, dout, q, false, 1, nullptr, nullptr, dP, true, st)) return cuda_fail("dp pass");
    if (launch_reverse_scan(f(L.ShB), f(L.Shend), p.BH, p.H, p.nseg, E, gamma, p.n, p.W, p.seg_chunks, 1, st))
        return cuda_fail("Sh scan");
    a.summary = nullptr;
    // B3: dv = RLA_{g^2}(p, q, dO), carry Zh (the transposed Zh^T)
    a.pow = 2;
    a.carry = f(L.Zhend);
    a.carry_mode = 1;
    if (fo_out(a, p.d, P, q, dout, false, 0, nullptr, nullptr, dvv, true, st)) return cuda_fail("dv pass");
    // B4: dk = RLA_g(k, dp, q) + RLA_g(k, q, dp), carry Sh + Sh^T
    a.pow = 1;
    a.carry = f(L.Shend);
    a.carry_mode = 2;
    if (fo_out(a, p.d, k, dP, q, true, 0, nullptr, nullptr, dk, true, st)) return cuda_fail("dk pass");
    // B5a: Z dO = LA_{g^2}(dO, v, p), carry Z^T;  B5b: dq = LA_g(dp, k, k) + that, carry S
    a.pow = 2;
    a.carry = f(L.Zin);
    a.carry_mode = 1;
    if (fo_out(a, p.d, dout, v, P, false, 0, nullptr, nullptr, dqa, false, st)) return cuda_fail("dq pass (Z dO)");
    a.pow = 1;
    a.carry = f(L.Sin);
    a.carry_mode = 0;
    if (fo_out(a, p.d, dP, k, nullptr, false, 0, nullptr, dqa, dq, false, st)) return cuda_fail("dq pass");
    return HLA2_OK;
}

size_t fo_forward_ws(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize, bool want_final) {
    const DevInfo di = dev_info();
    if (d != 128 || !fo_path(dtype, d, dv, chunk, normalize, di)) return 0;  // d = 64: the stored-p kernels
    const Plan p = fo_plan(B, H, n, d, di);
    if (p.nseg <= 0) return 0;
    const FoLayout L = fo_layout(p);
    return want_final ? L.final_total : L.fwd_total;
}

// The state after the last token from the first-order scans, once the forward part has formed
// the (q, v) summaries and the m and y moments (y from the stored full p): the carries of C, m, y
// into the last segment, and the last segment's combine with G = S C - Z and h = S m - y.
int fo_final_state(const Plan& p, const float* gamma, char* ws, const FoLayout& L, float* final_state,
                   cudaStream_t st) {
    auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t E = (size_t)p.d * p.d;
    const int seg_tokens = p.seg_chunks * p.W;
    // (one segment: the final-state kernel reads no carries)
    if (p.nseg > 1 && cudaMemsetAsync(ws + L.Cl, 0, L.carries_bytes, st) != cudaSuccess) return cuda_fail("carry reset");
    if (p.nseg > 1) {  // C, m and y carried into the last segment, in one launch
        const size_t dz = (size_t)p.d;
        const ScanJob jobs[3] = {{f(L.CB), f(L.Cl), E, p.nseg * E, E, 0, 1},
                                 {f(L.mB), f(L.ml), dz, p.nseg * dz, dz, 0, 1},
                                 {f(L.yB), f(L.yl), dz, p.nseg * dz, dz, 0, 2}};
        if (launch_linear_scans(jobs, 3, p.BH, p.H, p.nseg - 1, gamma, seg_tokens, st))
            return cuda_fail("last-segment carries");
    }
    FoFinal fin{};
    fin.SB = f(L.SB);
    fin.Sin = f(L.Sin);
    fin.ZB = f(L.ZB);
    fin.Zin = f(L.Zin);
    fin.CB = f(L.CB);
    fin.Cl = f(L.Cl);
    fin.ml = f(L.ml);
    fin.yl = f(L.yl);
    fin.mB = f(L.mB);
    fin.yB = f(L.yB);
    fin.BH = p.BH;
    fin.H = p.H;
    fin.n = p.n;
    fin.d = p.d;
    fin.nseg = p.nseg;
    fin.seg_tokens = seg_tokens;
    fin.gamma = gamma;
    if (launch_fo_final_state(fin, final_state, st)) return cuda_fail("final state");
    return HLA2_OK;
}

int fo_forward_call(const void* q, const void* k, const void* v, void* out, int B, int H, int n, const float* gamma,
                    cudaStream_t st, const hla2_opts* opts) {
    const DevInfo di = dev_info();
    const Plan p = fo_plan(B, H, n, 128, di);
    const FoLayout L = fo_layout(p);
    const bool want_final = opts->final_state != nullptr;
    const size_t need = want_final ? L.final_total : L.fwd_total;
    if (!opts->workspace || opts->workspace_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    char* ws = static_cast<char*>(opts->workspace);
    auto mark = [&](int i) {
        if (opts->phase_events && i < opts->n_phase_events && opts->phase_events[i] &&
            cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[i]), st) != cudaSuccess)
            cudaGetLastError();
    };
    cudaGetLastError();
    mark(0);
    // (d = 128 only: the final state's summaries come from the forward part's (p, v) pass)
    int rc = fo_forward_part(q, k, v, p, gamma, ws, L, st, want_final);
    mark(3);
    if (rc == HLA2_OK) rc = fo_output_pass(q, v, out, p, gamma, ws, L, st);
    mark(4);
    if (rc == HLA2_OK && want_final) rc = fo_final_state(p, gamma, ws, L, opts->final_state, st);
    mark(5);
    return rc == HLA2_OK ? succeed() : rc;
}

int check_backward(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize) {
    int rc = check_common(B, H, n, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    if (dtype == HLA2_BF16 && d != dv && !normalize)
        return fail(HLA2_ERR_UNSUPPORTED, "the bf16 backward needs d == dv (float32 takes any d, dv)");
    return HLA2_OK;
}

// Workspace of the ratio-normalised backward.  num and den are the unnormalised outputs of
// one recurrence for the widened value rows [v | e_0] (dv + kUnitWidth columns, column dv
// the unit), so one float32 unnormalised backward at that width covers both: its forward part
// writes [num | den], the quotient rule forms the upstream gradient [dL/dnum | dL/dden], and its
// reverse part gives dq, dk and [dv | .].  Its gradient is the difference of a numerator part
// and a denominator part that can each be tens of times larger than the result, hence float32.
// Layout: that backward's workspace, then float32 [B, H, n, *] buffers: the widened values,
// [num | den], the upstream gradient and [dv | .] (dv + kUnitWidth wide); for bf16 inputs
// also float32 copies of q, k and the float32 dq, dk (d wide).
constexpr int kUnitWidth = 16;
enum NormBuf { NB_VE, NB_ND, NB_DND, NB_DVE, NB_Q, NB_K, NB_DQ, NB_DK, NB_COUNT };
struct NormBwdLayout {
    BwdPlan bp;
    size_t buf[NB_COUNT] = {};
    size_t total = 0;
};

size_t unnormalised_backward_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype, const DevInfo& di) {
    if (fo_path(dtype, d, dv, chunk, 0, di)) {
        const Plan p = fo_plan(B, H, n, d, di);
        return p.nseg > 0 ? fo_layout(p).total : 0;
    }
    const BwdPlan bp = backward_plan(B, H, n, d, dv, chunk, dtype, di);
    if (!bp.W) return (size_t)-1;
    return bp.p.nseg > 0 ? bp.L.total_bytes : 0;
}

NormBwdLayout norm_bwd_layout(int B, int H, int n, int d, int dv, int chunk, int dtype, const DevInfo& di) {
    NormBwdLayout L;
    const int w = dv + kUnitWidth;
    L.bp = backward_plan(B, H, n, d, w, chunk, HLA2_F32, di);
    if (!L.bp.W) {
        L.total = (size_t)-1;
        return L;
    }
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t rows = (size_t)B * H * (size_t)n;
    const int width[NB_COUNT] = {w, w, w, w, d, d, d, d};
    const int count = dtype == HLA2_BF16 ? NB_COUNT : NB_Q;
    size_t o = up(L.bp.p.nseg > 0 ? L.bp.L.total_bytes : 0);
    for (int i = 0; i < count; ++i) {
        L.buf[i] = o;
        o += up(rows * (size_t)width[i] * sizeof(float));
    }
    L.total = o;
    return L;
}

int forward_saving_for_backward(const void* q, const void* k, const void* v, void* out, int B, int H, int n, int d,
                                int dv, const float* gamma, int normalize, int chunk, cudaStream_t st,
                                const hla2_opts* opts) {
    if (opts->dtype != HLA2_BF16 || d != dv || normalize || opts->init_state || opts->final_state)
        return fail(HLA2_ERR_UNSUPPORTED,
                    "saving for the backward needs bf16, d == dv, normalize == 0 and no init_state / final_state");
    const DevInfo di = dev_info();
    if (fo_path(opts->dtype, d, dv, chunk, normalize, di)) {
        const Plan p = fo_plan(B, H, n, d, di);
        const FoLayout L = fo_layout(p);
        if (!opts->workspace || opts->workspace_bytes < L.total)
            return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required to save for the backward (got %zu)",
                        L.total, opts->workspace ? opts->workspace_bytes : (size_t)0);
        if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        char* ws = static_cast<char*>(opts->workspace);
        cudaGetLastError();
        int rc = fo_forward_part(q, k, v, p, gamma, ws, L, st);
        if (rc == HLA2_OK) rc = fo_output_pass(q, v, out, p, gamma, ws, L, st);
        return rc == HLA2_OK ? succeed() : rc;
    }
    const int W = backward_width(d, chunk, di);
    if (!W) return fail(HLA2_ERR_UNSUPPORTED, "no backward kernel for d %d, chunk %d", d, chunk);
    const Plan p = make_plan(B, H, n, d, dv, W, di.sms, backward_per_sm(d, W, di));
    const BwdLayout L = bwd_layout(p);
    if (!opts->workspace || opts->workspace_bytes < L.total_bytes)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required to save for the backward (got %zu)",
                    L.total_bytes, opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const ChunkArgs a = backward_chunk_args(q, k, v, out, (long)B * H, H, n, p, gamma, opts->workspace, L);
    const std::function<void(int)> mark = [&](int i) {
        if (opts->phase_events && i < opts->n_phase_events && opts->phase_events[i] &&
            cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[i]), st) != cudaSuccess)
            cudaGetLastError();
    };
    cudaGetLastError();
    mark(0);
    const int rc = backward_forward_part(a, p, L, d, dv, kOutStates, st, &mark);
    if (rc != HLA2_OK) return rc;
    mark(5);
    return succeed();
}

}  // namespace

extern "C" {

size_t hla2_backward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize) {
    if (check_backward(B, H, n, d, dv, chunk, dtype, normalize) != HLA2_OK) return (size_t)-1;
    const DevInfo di = dev_info();
    if (normalize) return norm_bwd_layout(B, H, n, d, dv, chunk, dtype, di).total;
    return unnormalised_backward_bytes(B, H, n, d, dv, chunk, dtype, di);
}

int hla2_backward(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                  void* dv_out, int B, int H, int n, int d, int dv, const float* gamma, int normalize,
                  int chunk, hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_backward");
    if (!opts) return fail(HLA2_ERR_INVALID_ARG, "opts must not be NULL");
    int rc = check_backward(B, H, n, d, dv, chunk, opts->dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (opts->init_state || opts->final_state)
        return fail(HLA2_ERR_INVALID_ARG, "the backward takes no init_state / final_state");
    if (opts->flags & ~HLA2_FLAG_STATES_SAVED) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_backward");
    const long BH = (long)B * H;
    if (BH == 0 || n == 0) return succeed();
    if (!q || !k || !v || !dout || !dq || !dk || !dv_out)
        return fail(HLA2_ERR_INVALID_ARG, "q, k, v, dout, dq, dk, dv must not be NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv_out))
        return fail(HLA2_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    const DevInfo di = dev_info();
    if (normalize) {
        if (opts->flags & HLA2_FLAG_STATES_SAVED)
            return fail(HLA2_ERR_UNSUPPORTED, "saved forward states cover the unnormalised output only");
        if (!isfinite(opts->eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
        const NormBwdLayout N = norm_bwd_layout(B, H, n, d, dv, chunk, opts->dtype, di);
        if (N.total == (size_t)-1) return fail(HLA2_ERR_UNSUPPORTED, "no backward kernel for d %d, chunk %d", d, chunk);
        if (!opts->workspace || opts->workspace_bytes < N.total)
            return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", N.total,
                        opts->workspace ? opts->workspace_bytes : (size_t)0);
        if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        char* base = static_cast<char*>(opts->workspace);
        auto buf = [&](int i) { return reinterpret_cast<float*>(base + N.buf[i]); };
        const bool bf = opts->dtype == HLA2_BF16;
        const size_t rows = (size_t)BH * (size_t)n;
        const int w = dv + kUnitWidth;
        const BwdPlan& bp = N.bp;
        cudaStream_t s2 = reinterpret_cast<cudaStream_t>(stream);
        cudaGetLastError();
        const float* q32 = bf ? buf(NB_Q) : static_cast<const float*>(q);
        const float* k32 = bf ? buf(NB_K) : static_cast<const float*>(k);
        float* dq32 = bf ? buf(NB_DQ) : static_cast<float*>(dq);
        float* dk32 = bf ? buf(NB_DK) : static_cast<float*>(dk);
        if (bf && (launch_convert_bf16_f32(static_cast<const bf16*>(q), buf(NB_Q), rows * d, s2) ||
                   launch_convert_bf16_f32(static_cast<const bf16*>(k), buf(NB_K), rows * d, s2)))
            return cuda_fail("float32 copies");
        if (launch_widen_values(v, buf(NB_VE), rows, dv, w, bf, s2)) return cuda_fail("widened values");
        // [num | den] and the states the reverse passes read
        const ChunkArgs a = backward_chunk_args(q32, k32, buf(NB_VE), nullptr, BH, H, n, bp.p, gamma, base, bp.L);
        if ((rc = backward_forward_part_f32(a, bp.p, bp.L, d, w, s2, buf(NB_ND))) != HLA2_OK) return rc;
        if (launch_quotient_rule(dout, buf(NB_ND), buf(NB_DND), rows, dv, w, opts->eps, bf, s2))
            return cuda_fail("quotient rule");
        if ((rc = backward_reverse_part_f32(q32, k32, buf(NB_VE), buf(NB_DND), dq32, dk32, buf(NB_DVE), H, bp.p, bp.L,
                                            gamma, reinterpret_cast<float*>(base), d, w, s2)) != HLA2_OK)
            return rc;
        if (launch_narrow_values(buf(NB_DVE), dv_out, rows, dv, w, bf, s2)) return cuda_fail("value gradient");
        if (bf && (launch_convert_f32_bf16(dq32, static_cast<bf16*>(dq), rows * d, s2) ||
                   launch_convert_f32_bf16(dk32, static_cast<bf16*>(dk), rows * d, s2)))
            return cuda_fail("bf16 gradients");
        return succeed();
    }
    if (fo_path(opts->dtype, d, dv, chunk, 0, di)) {
        const Plan p = fo_plan(B, H, n, d, di);
        const FoLayout L = fo_layout(p);
        if (!opts->workspace || opts->workspace_bytes < L.total)
            return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", L.total,
                        opts->workspace ? opts->workspace_bytes : (size_t)0);
        if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        char* ws = static_cast<char*>(opts->workspace);
        cudaStream_t sf = reinterpret_cast<cudaStream_t>(stream);
        cudaGetLastError();
        if (opts->flags & HLA2_FLAG_STATES_SAVED) {
            if (cudaMemsetAsync(ws, 0, sizeof(int), sf) != cudaSuccess) return cuda_fail("status word");
        } else if ((rc = fo_forward_part(q, k, v, p, gamma, ws, L, sf)) != HLA2_OK) {
            return rc;
        }
        rc = fo_reverse_part(q, k, v, dout, dq, dk, dv_out, p, gamma, ws, L, sf);
        return rc == HLA2_OK ? succeed() : rc;
    }
    const BwdPlan bp = backward_plan(B, H, n, d, dv, chunk, opts->dtype, di);
    if (!bp.W) return fail(HLA2_ERR_UNSUPPORTED, "no backward kernel for d %d, dv %d, chunk %d", d, dv, chunk);
    if (bp.f32 && (opts->flags & HLA2_FLAG_STATES_SAVED))
        return fail(HLA2_ERR_UNSUPPORTED, "saved forward states are kept by the bf16 path only");
    if (!opts->workspace || opts->workspace_bytes < bp.L.total_bytes)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", bp.L.total_bytes,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    if (bp.f32) {
        cudaStream_t sf = reinterpret_cast<cudaStream_t>(stream);
        cudaGetLastError();
        const ChunkArgs a = backward_chunk_args(q, k, v, nullptr, BH, H, n, bp.p, gamma, opts->workspace, bp.L);
        if ((rc = backward_forward_part_f32(a, bp.p, bp.L, d, dv, sf)) != HLA2_OK) return rc;
        if ((rc = backward_reverse_part_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                            static_cast<const float*>(v), static_cast<const float*>(dout),
                                            static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv_out),
                                            H, bp.p, bp.L, gamma, static_cast<float*>(opts->workspace), d, dv, sf)) !=
            HLA2_OK)
            return rc;
        return succeed();
    }
    const int W = bp.W;
    const Plan& p = bp.p;
    const BwdLayout& L = bp.L;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* ws = static_cast<float*>(opts->workspace);
    bf16* states = reinterpret_cast<bf16*>(static_cast<char*>(opts->workspace) + L.states_bytes_off);

    const ChunkArgs a = backward_chunk_args(q, k, v, nullptr, BH, H, n, p, gamma, opts->workspace, L);

    BwdArgs b{};
    b.q = static_cast<const bf16*>(q);
    b.k = static_cast<const bf16*>(k);
    b.v = static_cast<const bf16*>(v);
    b.dout = static_cast<const bf16*>(dout);
    b.dq = static_cast<bf16*>(dq);
    b.dk = static_cast<bf16*>(dk);
    b.dv = static_cast<bf16*>(dv_out);
    b.BH = (int)BH;
    b.H = H;
    b.n = n;
    b.W = W;
    b.nchunks = p.nchunks;
    b.seg_chunks = p.seg_chunks;
    b.nseg = p.nseg;
    b.gamma = gamma;
    b.ws = ws;
    b.ZhB = L.ZhB;
    b.ShB = L.ShB;
    b.Zh_end = L.Zh_end;
    b.Sh_end = L.Sh_end;
    b.chunk_states = states;

    const size_t dd = (size_t)d * d, ddv = (size_t)d * dv;
    cudaGetLastError();
    if (!(opts->flags & HLA2_FLAG_STATES_SAVED)) {
        rc = backward_forward_part(a, p, L, d, dv, kStates, st, nullptr);
        if (rc != HLA2_OK) return rc;
    }
    // reverse summaries, reverse scan with the cross term Zh_end C_B^T, gradients
    if (launch_bwd_chunk_mma(b, d, W, true, st)) return cuda_fail("reverse summaries");
    if (launch_reverse_scan(ws + L.ZhB, ws + L.Zh_end, a.BH, H, p.nseg, ddv, gamma, n, W, p.seg_chunks, 2, st) ||
        launch_reverse_cross(b, ws + L.F.CB, d, dv, st) ||
        launch_reverse_scan(ws + L.ShB, ws + L.Sh_end, a.BH, H, p.nseg, dd, gamma, n, W, p.seg_chunks, 1, st))
        return cuda_fail("reverse segment scan");
    if (launch_bwd_chunk_mma(b, d, W, false, st)) return cuda_fail("gradient pass");
    return succeed();
}

int hla2_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H,
                     int d, int dv, const float* gamma, int normalize, hla2_stream_t stream,
                     const hla2_opts* opts) {
    NvtxScope nvtx("hla2_decode_step");
    const int dtype = opts ? opts->dtype : HLA2_BF16;
    const float eps = opts ? opts->eps : 1e-6f;
    const int flags = opts ? opts->flags : 0;
    int rc = check_common(N, H, 0, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (normalize && !isfinite(eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (flags & ~(HLA2_FLAG_COMPACT_STATE | HLA2_FLAG_UNMASKED))
        return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_decode_step");
    if ((long)N * H == 0) return succeed();
    if (!state || !q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "state, q, k, v, out must not be NULL");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    cudaGetLastError();
    if (launch_decode_step(state, q, k, v, out, N, H, d, dv, gamma, normalize, eps, dtype == HLA2_BF16,
                           (flags & HLA2_FLAG_COMPACT_STATE) != 0, (flags & HLA2_FLAG_UNMASKED) != 0,
                           reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("decode step");
    return succeed();
}

int hla2_decode_step_mq(float* key_state, float* head_state, const void* q, const void* k, const void* v,
                        void* out, int N, int Hk, int group, int d, int dv, const float* gamma, int normalize,
                        hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_decode_step_mq");
    const int dtype = opts ? opts->dtype : HLA2_BF16;
    const float eps = opts ? opts->eps : 1e-6f;
    const int flags = opts ? opts->flags : 0;
    int rc = check_common(N, Hk, 0, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (group < 1 || group > 8) return fail(HLA2_ERR_INVALID_ARG, "group must be 1 to 8 query heads per key (got %d)", group);
    if (normalize && !isfinite(eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (flags & HLA2_FLAG_COMPACT_STATE)
        return fail(HLA2_ERR_UNSUPPORTED, "the multi-query step keeps the shared S in the packed layout");
    if (flags & ~HLA2_FLAG_UNMASKED) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_decode_step_mq");
    if ((long)N * Hk == 0) return succeed();
    if (!key_state || !head_state || !q || !k || !v || !out)
        return fail(HLA2_ERR_INVALID_ARG, "state, q, k, v, out must not be NULL");
    if (!aligned16(key_state) || !aligned16(head_state) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    cudaGetLastError();
    if (launch_decode_mq(key_state, head_state, q, k, v, out, N, Hk, group, d, dv, gamma, normalize, eps,
                         dtype == HLA2_BF16, (flags & HLA2_FLAG_UNMASKED) != 0, reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("multi-query decode step");
    return succeed();
}

size_t hla2_mq_head_state_floats(int d, int dv) { return 2 * (size_t)d * dv + 2 * (size_t)d; }

int hla2_hla3_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H, int d,
                          int dv, int normalize, hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_hla3_decode_step");
    const int dtype = opts ? opts->dtype : HLA2_BF16;
    const float eps = opts ? opts->eps : 1e-6f;
    int rc = check_common(N, H, 0, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (normalize && !isfinite(eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (opts && opts->flags) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_hla3_decode_step");
    if ((long)N * H == 0) return succeed();
    if (!state || !q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "state, q, k, v, out must not be NULL");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    cudaGetLastError();
    if (launch_hla3_decode_step(state, q, k, v, out, (long)N * H, d, dv, normalize, eps, dtype == HLA2_BF16,
                                reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("third-order decode step");
    return succeed();
}

size_t hla2_compact_state_floats(int d, int dv) { return compact_state_floats(d, dv); }

size_t hla2_ahla_state_floats(int d, int dv) { return ahla_state_floats(d, dv); }

int hla2_ahla_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H, int d,
                          int dv, const float* gamma, int normalize, hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_ahla_decode_step");
    const int dtype = opts ? opts->dtype : HLA2_BF16;
    const float eps = opts ? opts->eps : 1e-6f;
    int rc = check_common(N, H, 0, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (normalize && !isfinite(eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (opts && opts->flags) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_ahla_decode_step");
    if ((long)N * H == 0) return succeed();
    if (!state || !q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "state, q, k, v, out must not be NULL");
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    cudaGetLastError();
    if (launch_ahla_decode_step(state, q, k, v, out, N, H, d, dv, gamma, normalize, eps, dtype == HLA2_BF16,
                                reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("AHLA decode step");
    return succeed();
}

static int ahla_check(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize) {
    int rc = check_common(B, H, n, d, dv, dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    const bool tc = chunk == 128 && d == 64 && !normalize;
    if (dtype != HLA2_BF16 || d != dv || (chunk != 32 && chunk != 64 && !tc))
        return fail(HLA2_ERR_UNSUPPORTED,
                    "the AHLA forward covers bf16, d == dv and chunk 32 or 64 (chunk 128: d = 64, unnormalised)");
    if (tc && !ahla_tc_available()) return fail(HLA2_ERR_UNSUPPORTED, "tensor-map encoding is not available");
    return HLA2_OK;
}

// chunk 128 runs the tcgen05 kernel, chunks 32 and 64 the mma.sync one
// ---- masked third-order output (gamma = 1): first-order pass, then the second-order forward ----

static Plan ahla_plan(int B, int H, int n, int d, int chunk);

// The first-order pass runs on the AHLA tcgen05 kernel in its first-order mode (Inner is the
// masked first-order output) for bf16, d = dv = 64; elsewhere on the SIMT kernel.
static bool hla3_first_order_on_tc(bool bf, int d, int w, const DevInfo& di) {
    return bf && d == 64 && w == 64 && !tc_disabled() && ahla_tc_available() && ahla_tc_smem() <= (size_t)di.smem_optin;
}

static constexpr int kHla3Unit = 16;  // value width of the denominator passes (column 0 is 1)

static int hla3_la_width(int d, int dv, int chunk, const DevInfo& di) {
    for (int W = chunk < 64 ? chunk : 64; W >= 16; W /= 2)
        if (first_order_smem(d, dv, W) <= (size_t)di.smem_optin &&
            first_order_smem(d, kHla3Unit, W) <= (size_t)di.smem_optin)
            return W;
    return 0;
}

// Chunk width of the third-order output's second-order passes: the largest <= chunk with a
// forward kernel for both value widths (the result does not depend on the width).
static int hla3_second_width(int dtype, int d, int dv, int chunk, int normalize, const DevInfo& di) {
    for (int W = chunk; W >= 16; W /= 2)
        if (choose_forward_path(dtype, d, dv, W, 0, false, di) != Path::kNone &&
            (!normalize || choose_forward_path(dtype, d, kHla3Unit, W, 0, false, di) != Path::kNone))
            return W;
    return 0;
}

// u = LA(q, k, v) on the d = 64 first-order scan kernels (bf16, d = w = 64, no first-order final
// state): the (k, v) summaries of every segment, their prefix over the segments, one output
// pass.  Workspace: the status word, then the summaries and the carries, [BH][nseg][64*64] fp32.
static bool hla3_first_order_on_fo(bool bf, int d, int w, const float* final_P, const DevInfo& di) {
    return bf && d == 64 && w == 64 && !final_P && fo_path(HLA2_BF16, 64, 64, 128, 0, di);
}
static size_t hla3_fo_bytes(int B, int H, int n, const DevInfo& di) {
    const Plan p = fo_plan(B, H, n, 64, di);
    return 256 + 2 * (size_t)p.BH * p.nseg * 64 * 64 * sizeof(float);
}

struct Hla3Layout {
    int W = 0;
    int W2 = 0;  // chunk width of the second-order passes
    Plan p;
    size_t PB = 0, Pin = 0;  // first-order workspace (floats, in the scratch region)
    size_t scratch = 0;      // bytes of the scratch region (first-order and second-order calls in turn)
    size_t u = 0, e0 = 0, u1 = 0, den = 0;  // byte offsets
    size_t pk_num = 0, pk_den = 0, p_num = 0, p_den = 0;  // final-state pieces (byte offsets)
    size_t total = 0;
};

static Hla3Layout hla3_layout(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize,
                              bool want_final, const DevInfo& di) {
    Hla3Layout L;
    const bool dens = normalize || want_final;  // the unit-value passes run
    L.W = hla3_la_width(d, dv, chunk, di);
    L.W2 = hla3_second_width(dtype, d, dv, chunk, dens, di);
    if (!L.W || !L.W2) {
        L.W = 0;
        return L;
    }
    chunk = L.W2;
    L.p = make_plan(B, H, n, d, dv, L.W, di.sms, blocks_per_sm(first_order_smem(d, dv, L.W), 256, 4, di));
    const size_t BH = (size_t)B * H, ns = L.p.nseg, nsm = ns > 0 ? ns - 1 : 0;
    const size_t wmax = dv > kHla3Unit ? dv : kHla3Unit;
    L.PB = kStatusFloats;
    L.Pin = align64(L.PB + BH * nsm * (size_t)d * wmax);
    size_t la = align64(L.Pin + BH * ns * (size_t)d * wmax) * sizeof(float);
    if (hla3_first_order_on_tc(dtype == HLA2_BF16, d, dv, di)) {
        const size_t t = ahla_layout(ahla_plan(B, H, n, d, 128)).total * sizeof(float);
        la = la > t ? la : t;
    }
    if (dtype == HLA2_BF16 && d == 64 && dv == 64) {  // the first-order pass on the d = 64 scan kernels
        const size_t t = hla3_fo_bytes(B, H, n, di);
        la = la > t ? la : t;
    }
    size_t f1 = hla2_forward_workspace_bytes(B, H, n, d, dv, chunk, dtype, 0, want_final);
    size_t f2 = dens ? hla2_forward_workspace_bytes(B, H, n, d, kHla3Unit, chunk, dtype, 0, want_final) : 0;
    if (f1 == (size_t)-1 || f2 == (size_t)-1) {
        L.W = 0;
        return L;
    }
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    L.scratch = up(la > f1 ? (la > f2 ? la : f2) : (f1 > f2 ? f1 : f2));
    const size_t es = dtype == HLA2_BF16 ? 2 : 4, rows = BH * (size_t)n;
    size_t o = L.scratch;
    L.u = o;
    o += up(rows * dv * es);
    if (dens) {
        L.e0 = o;
        o += up(rows * kHla3Unit * es);
        L.u1 = o;
        o += up(rows * kHla3Unit * es);
        L.den = o;
        o += up(rows * kHla3Unit * es);
    }
    if (want_final) {
        const size_t dd = (size_t)d * d;
        L.pk_num = o;
        o += up(BH * (dd + 2 * (size_t)d * dv + 2 * (size_t)d) * sizeof(float));
        L.pk_den = o;
        o += up(BH * (dd + 2 * (size_t)d * kHla3Unit + 2 * (size_t)d) * sizeof(float));
        L.p_num = o;
        o += up(BH * (size_t)d * dv * sizeof(float));
        L.p_den = o;
        o += up(BH * (size_t)d * kHla3Unit * sizeof(float));
    }
    L.total = o;
    return L;
}

extern "C" size_t hla2_hla3_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                                    int normalize, int want_final_state) {
    if (check_common(B, H, n, d, dv, dtype, normalize) != HLA2_OK || !dim_ok(chunk)) return (size_t)-1;
    const Hla3Layout L = hla3_layout(B, H, n, d, dv, chunk, dtype, normalize, want_final_state != 0, dev_info());
    return L.W ? L.total : (size_t)-1;
}

// first-order pass u = masked linear attention (q, k, values) into `u`
static int hla3_first_order(const void* q, const void* k, const void* vals, void* u, int B, int H, int n, int d,
                            int w, const Hla3Layout& L, void* ws, bool bf, cudaStream_t st, float* final_P) {
    const DevInfo di = dev_info();
    if (hla3_first_order_on_fo(bf, d, w, final_P, di)) {
        const Plan pf = fo_plan(B, H, n, 64, di);
        char* wsb = static_cast<char*>(ws);
        const size_t E = 64 * 64;
        float* SB = reinterpret_cast<float*>(wsb + 256);
        float* Sin = SB + (size_t)pf.BH * pf.nseg * E;
        FoArgs a = fo_args(pf, nullptr, wsb);
        a.pow = 1;
        a.summary = SB;
        if (launch_fo_zero_first(Sin, pf.BH, pf.nseg, (int)E, a.status, st)) return cuda_fail("first-order carry-in");
        if (fo_summary(a, 64, k, vals, false, st)) return cuda_fail("first-order summaries");
        if (pf.nseg > 1 && launch_linear_scan(SB, Sin, pf.BH, pf.H, pf.nseg - 1, E, pf.nseg * E, pf.nseg * E, true,
                                              nullptr, pf.seg_chunks * pf.W, 1, st))
            return cuda_fail("first-order scan");
        a.carry = Sin;
        a.carry_mode = 0;
        return fo_out(a, 64, q, k, vals, false, 0, nullptr, nullptr, u, false, st) ? cuda_fail("first-order pass")
                                                                                  : HLA2_OK;
    }
    if (hla3_first_order_on_tc(bf, d, w, di)) {
        const Plan p = ahla_plan(B, H, n, d, 128);
        AhlaArgs a{};
        a.q = q;
        a.k = k;
        a.v = vals;
        a.out = u;
        a.BH = B * H;
        a.H = H;
        a.n = n;
        a.W = 128;
        a.nchunks = p.nchunks;
        a.seg_chunks = p.seg_chunks;
        a.nseg = p.nseg;
        a.nsum = p.nseg - 1;
        a.ws = static_cast<float*>(ws);
        a.L = ahla_layout(p);
        a.final_state = final_P;  // first-order mode: P only, [BH][d*d]
        int* status = static_cast<int*>(ws);
        if (launch_ahla_init(a, d, st)) return cuda_fail("first-order carry-in");
        if (p.nseg > 1) {
            AhlaArgs b = a;
            b.seg0 = 0;
            b.nseg_launch = p.nseg - 1;
            if (launch_ahla_tc(b, true, status, st, true)) return cuda_fail("first-order summaries");
            const size_t dd = (size_t)d * d;
            if (launch_linear_scan(a.ws + a.L.PB, a.ws + a.L.Pin, a.BH, H, p.nseg - 1, dd, a.nsum * dd, p.nseg * dd,
                                   true, nullptr, p.seg_chunks * 128, 1, st))
                return cuda_fail("first-order scan");
        }
        AhlaArgs b = a;
        b.seg0 = 0;
        b.nseg_launch = p.nseg;
        return launch_ahla_tc(b, false, status, st, true) ? cuda_fail("first-order pass") : HLA2_OK;
    }
    LaArgs a{};
    a.q = q;
    a.k = k;
    a.v = vals;
    a.u = u;
    a.BH = B * H;
    a.H = H;
    a.n = n;
    a.d = d;
    a.dv = w;
    a.W = L.W;
    a.nchunks = L.p.nchunks;
    a.seg_chunks = L.p.seg_chunks;
    a.nseg = L.p.nseg;
    a.gamma = nullptr;
    a.ws = static_cast<float*>(ws);
    a.PB = L.PB;
    a.Pin = L.Pin;
    a.final_P = final_P;
    return launch_first_order_forward(a, bf, st) ? cuda_fail("first-order pass") : HLA2_OK;
}

extern "C" int hla2_hla3_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n, int d,
                                 int dv, const float* gamma, int normalize, int chunk, hla2_stream_t stream,
                                 const hla2_opts* opts) {
    NvtxScope nvtx("hla2_hla3_forward");
    if (!opts) return fail(HLA2_ERR_INVALID_ARG, "opts must not be NULL");
    int rc = check_common(B, H, n, d, dv, opts->dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    if (normalize && !isfinite(opts->eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (opts->flags) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_hla3_forward");
    if (gamma) return fail(HLA2_ERR_UNSUPPORTED, "the third-order scan is defined for gamma = 1 (pass NULL)");
    if (opts->init_state) return fail(HLA2_ERR_UNSUPPORTED, "the third-order forward starts from the empty prefix");
    const bool want_final = opts->final_state != nullptr;
    if (want_final && !aligned16(opts->final_state))
        return fail(HLA2_ERR_INVALID_ARG, "final_state must be 16-byte aligned");
    if ((long)B * H == 0) return succeed();
    if (n == 0) {
        if (want_final && cudaMemsetAsync(opts->final_state, 0, (size_t)B * H * raw_state_floats(d, dv) * sizeof(float),
                                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return cuda_fail("final state");
        return succeed();
    }
    if (!q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must not be NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
    const DevInfo di = dev_info();
    const Hla3Layout L = hla3_layout(B, H, n, d, dv, chunk, opts->dtype, normalize, want_final, di);
    if (!L.W) return fail(HLA2_ERR_UNSUPPORTED, "no kernel for d %d, dv %d, chunk %d", d, dv, chunk);
    if (!opts->workspace || opts->workspace_bytes < L.total)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", L.total,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(opts->workspace);
    const bool bf = opts->dtype == HLA2_BF16;
    hla2_opts so{};
    so.dtype = opts->dtype;
    so.eps = opts->eps;
    so.workspace = base;
    so.workspace_bytes = L.scratch;
    cudaGetLastError();
    auto fbuf = [&](size_t off) { return want_final ? reinterpret_cast<float*>(base + off) : nullptr; };
    // numerator: the masked second-order output with the first-order outputs as values
    if ((rc = hla3_first_order(q, k, v, base + L.u, B, H, n, d, dv, L, base, bf, st, fbuf(L.p_num))) != HLA2_OK)
        return rc;
    so.final_state = fbuf(L.pk_num);
    if ((rc = hla2_forward(q, k, base + L.u, out, B, H, n, d, dv, nullptr, 0, L.W2, stream, &so)) != HLA2_OK)
        return rc;
    if (normalize || want_final) {  // the same with v -> 1 (value rows e_0, column 0)
        const size_t rows = (size_t)B * H * n;
        if (launch_unit_rows(base + L.e0, rows, kHla3Unit, bf, st)) return cuda_fail("unit value rows");
        if ((rc = hla3_first_order(q, k, base + L.e0, base + L.u1, B, H, n, d, kHla3Unit, L, base, bf, st,
                                   fbuf(L.p_den))) != HLA2_OK)
            return rc;
        so.final_state = fbuf(L.pk_den);
        if ((rc = hla2_forward(q, k, base + L.u1, base + L.den, B, H, n, d, kHla3Unit, nullptr, 0, L.W2, stream,
                               &so)) != HLA2_OK)
            return rc;
        if (normalize && launch_divide_rows(out, base + L.den, rows, dv, kHla3Unit, opts->eps, bf, st))
            return cuda_fail("normalisation");
    }
    if (want_final && launch_hla3_assemble_state(opts->final_state, fbuf(L.pk_num), fbuf(L.pk_den), fbuf(L.p_num),
                                                 fbuf(L.p_den), (long)B * H, d, dv, kHla3Unit, st))
        return cuda_fail("final state");
    return succeed();
}

// ---- AHLA reverse mode ----------------------------------------------------------------------

static int ahla_bwd_width(int d, int chunk, const DevInfo& di) {
    for (int W = chunk < 32 ? chunk : 32; W >= 16; W /= 2)
        if (ahla_bwd_smem(d, W) <= (size_t)di.smem_optin) return W;
    return 0;
}

struct AhlaBwdPlan {
    int W = 0;
    Plan p;
    AhlaBwdLayout L;
};

static AhlaBwdPlan ahla_bwd_plan(int B, int H, int n, int d, int chunk, const DevInfo& di) {
    AhlaBwdPlan bp;
    bp.W = ahla_bwd_width(d, chunk, di);
    if (!bp.W) return bp;
    bp.p = make_plan(B, H, n, d, d, bp.W, di.sms, blocks_per_sm(ahla_bwd_smem(d, bp.W), 256, 4, di));
    bp.L = ahla_bwd_layout(B * H, bp.p.nseg, bp.p.nchunks, d);
    return bp;
}

// ---- AHLA reverse mode on the tcgen05 first-order scans (bf16, d = dv = 64, chunk >= 128) ------
// AHLA is two chained first-order scans with the same queries and keys, u = LA_g(q, k, v) and
// o = LA_g(q, k, u).  Its reverse mode:
//   du = RLA_g(k, q, dO),  dv = RLA_g(k, q, du),
//   dk = RLA_g(u, dO, q) + RLA_g(v, du, q),  dq = LA_g(dO, u, k) + LA_g(du, v, k),
// whose carries are four summaries (some read transposed): KV = sum k v^T (F1, forward),
// UK = sum u k^T (over the u pass's own output), QD = sum q dO^T (B1, reverse) and DQ =
// sum du q^T (over the du pass's own output).  dk and dq each take one pass over their two
// query / key pairs, which share the values.
struct AhlaFoLayout {
    size_t KVB, KVin, UKB, UKin, QDB, QDend, DQB, DQend;  // byte offsets, fp32 [BH][nseg][d][d]
    size_t U, DU;                                         // byte offsets, bf16 [BH][n][d]
    size_t total;
};

AhlaFoLayout ahla_fo_layout(const Plan& p) {
    AhlaFoLayout L;
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t sum = (size_t)p.BH * p.nseg * p.d * p.d * sizeof(float);
    const size_t tok = (size_t)p.BH * p.n * p.d * sizeof(bf16);
    size_t o = 256;  // status word
    size_t* sums[] = {&L.KVB, &L.KVin, &L.UKB, &L.UKin, &L.QDB, &L.QDend, &L.DQB, &L.DQend};
    for (size_t* x : sums) {
        *x = o;
        o = up(o + sum);
    }
    size_t* toks[] = {&L.U, &L.DU};
    for (size_t* x : toks) {
        *x = o;
        o = up(o + tok);
    }
    L.total = o;
    return L;
}

bool ahla_fo_path(int dtype, int d, int dv, int chunk, const DevInfo& di) {
    return d == 64 && fo_path(dtype, d, dv, chunk, 0, di);
}

int ahla_fo_backward(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk, void* dvv,
                     const Plan& p, const float* gamma, char* ws, const AhlaFoLayout& L, cudaStream_t st) {
    auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
    const size_t E = (size_t)p.d * p.d;
    const int seg_tokens = p.seg_chunks * p.W;
    void* U = ws + L.U;
    void* DU = ws + L.DU;
    FoArgs a = fo_args(p, gamma, ws);
    a.pow = 1;
    a.pow_next = 1;
    // F1: KV summaries and the forward scan
    a.summary = f(L.KVB);
    if (fo_summary(a, p.d, k, v, false, st)) return cuda_fail("AHLA key-value summaries");
    if (launch_fo_zero_first(f(L.KVin), p.BH, p.nseg, (int)E, a.status, st) ||
        (p.nseg > 1 && launch_linear_scan(f(L.KVB), f(L.KVin), p.BH, p.H, p.nseg - 1, E, p.nseg * E, p.nseg * E, true,
                                          gamma, seg_tokens, 1, st)))
        return cuda_fail("AHLA key-value scan");
    // F2: u = LA(q, k, v), UK summaries over (u, k)
    a.carry = f(L.KVin);
    a.carry_mode = 0;
    a.summary = f(L.UKB);
    if (fo_out(a, p.d, q, k, v, false, 2, k, nullptr, U, false, st)) return cuda_fail("AHLA u pass");
    if (launch_fo_zero_first(f(L.UKin), p.BH, p.nseg, (int)E, nullptr, st) ||
        (p.nseg > 1 && launch_linear_scan(f(L.UKB), f(L.UKin), p.BH, p.H, p.nseg - 1, E, p.nseg * E, p.nseg * E, true,
                                          gamma, seg_tokens, 1, st)))
        return cuda_fail("AHLA u-key scan");
    // B1: QD summaries (reverse) and the reverse scan
    a.carry = nullptr;
    a.summary = f(L.QDB);
    if (fo_summary(a, p.d, q, dout, true, st)) return cuda_fail("AHLA query-gradient summaries");
    if (launch_reverse_scan(f(L.QDB), f(L.QDend), p.BH, p.H, p.nseg, E, gamma, p.n, p.W, p.seg_chunks, 1, st))
        return cuda_fail("AHLA query-gradient scan");
    // B2: du = RLA(k, q, dO), DQ summaries over (du, q)
    a.carry = f(L.QDend);
    a.carry_mode = 0;
    a.summary = f(L.DQB);
    if (fo_out(a, p.d, k, q, dout, false, 2, q, nullptr, DU, true, st)) return cuda_fail("AHLA du pass");
    if (launch_reverse_scan(f(L.DQB), f(L.DQend), p.BH, p.H, p.nseg, E, gamma, p.n, p.W, p.seg_chunks, 1, st))
        return cuda_fail("AHLA du-query scan");
    a.summary = nullptr;
    // B3: dv = RLA(k, q, du), carry sum q du^T
    a.carry = f(L.DQend);
    a.carry_mode = 1;
    if (fo_out(a, p.d, k, q, DU, false, 0, nullptr, nullptr, dvv, true, st)) return cuda_fail("AHLA dv pass");
    // B4: dk = RLA(u, dO, q) [carry sum dO q^T] + RLA(v, du, q) [carry sum du q^T]
    a.carry = f(L.QDend);
    a.carry_mode = 1;
    a.carry2 = f(L.DQend);
    a.carry_mode2 = 0;
    if (launch_fo64_tc_out2(a, U, dout, v, DU, q, dk, true, st)) return cuda_fail("AHLA dk pass");
    // B5: dq = LA(dO, u, k) [carry sum u k^T] + LA(du, v, k) [carry sum v k^T]
    a.carry = f(L.UKin);
    a.carry_mode = 0;
    a.carry2 = f(L.KVin);
    a.carry_mode2 = 1;
    if (launch_fo64_tc_out2(a, dout, U, DU, v, k, dq, false, st)) return cuda_fail("AHLA dq pass");
    return HLA2_OK;
}

extern "C" size_t hla2_ahla_backward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                                     int normalize) {
    if (check_common(B, H, n, d, dv, dtype, normalize) != HLA2_OK || !dim_ok(chunk) || d != dv || normalize)
        return (size_t)-1;
    if (ahla_fo_path(dtype, d, dv, chunk, dev_info())) {
        const Plan p = fo_plan(B, H, n, d, dev_info());
        return p.nseg > 0 ? ahla_fo_layout(p).total : 0;
    }
    const AhlaBwdPlan bp = ahla_bwd_plan(B, H, n, d, chunk, dev_info());
    if (!bp.W) return (size_t)-1;
    return bp.p.nseg > 0 ? bp.L.total * sizeof(float) : 0;
}

extern "C" int hla2_ahla_backward(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                                  void* dv_out, int B, int H, int n, int d, int dv, const float* gamma, int normalize,
                                  int chunk, hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_ahla_backward");
    if (!opts) return fail(HLA2_ERR_INVALID_ARG, "opts must not be NULL");
    int rc = check_common(B, H, n, d, dv, opts->dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (!dim_ok(chunk)) return fail(HLA2_ERR_INVALID_ARG, "chunk must be 16, 32, 64 or 128 (got %d)", chunk);
    if (d != dv) return fail(HLA2_ERR_UNSUPPORTED, "the AHLA backward needs d == dv");
    if (normalize) return fail(HLA2_ERR_UNSUPPORTED, "the AHLA backward covers the unnormalised output");
    if (opts->flags || opts->init_state || opts->final_state)
        return fail(HLA2_ERR_INVALID_ARG, "the AHLA backward takes no flags, init_state or final_state");
    const long BH = (long)B * H;
    if (BH == 0 || n == 0) return succeed();
    if (!q || !k || !v || !dout || !dq || !dk || !dv_out)
        return fail(HLA2_ERR_INVALID_ARG, "q, k, v, dout, dq, dk, dv must not be NULL");
    const DevInfo di = dev_info();
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv_out))
        return fail(HLA2_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    if (ahla_fo_path(opts->dtype, d, dv, chunk, di)) {
        const Plan p = fo_plan(B, H, n, d, di);
        const AhlaFoLayout L = ahla_fo_layout(p);
        if (!opts->workspace || opts->workspace_bytes < L.total)
            return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", L.total,
                        opts->workspace ? opts->workspace_bytes : (size_t)0);
        if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        cudaGetLastError();
        rc = ahla_fo_backward(q, k, v, dout, dq, dk, dv_out, p, gamma, static_cast<char*>(opts->workspace), L,
                              reinterpret_cast<cudaStream_t>(stream));
        return rc == HLA2_OK ? succeed() : rc;
    }
    const AhlaBwdPlan bp = ahla_bwd_plan(B, H, n, d, chunk, di);
    if (!bp.W) return fail(HLA2_ERR_UNSUPPORTED, "no AHLA backward kernel for d %d", d);
    const size_t need = bp.L.total * sizeof(float);
    if (!opts->workspace || opts->workspace_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    AhlaBwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.dout = dout;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv_out;
    a.BH = (int)BH;
    a.H = H;
    a.n = n;
    a.d = d;
    a.W = bp.W;
    a.nchunks = bp.p.nchunks;
    a.seg_chunks = bp.p.seg_chunks;
    a.nseg = bp.p.nseg;
    a.gamma = gamma;
    a.ws = static_cast<float*>(opts->workspace);
    a.PB = bp.L.PB;
    a.EB = bp.L.EB;
    a.RB = bp.L.RB;
    a.Pin = bp.L.Pin;
    a.Ein = bp.L.Ein;
    a.EhB = bp.L.EhB;
    a.PhB = bp.L.PhB;
    a.Eh_end = bp.L.Eh_end;
    a.Ph_end = bp.L.Ph_end;
    a.states = bp.L.states;
    cudaGetLastError();
    if (launch_ahla_backward(a, opts->dtype == HLA2_BF16, reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("AHLA backward");
    return succeed();
}

static Plan ahla_plan(int B, int H, int n, int d, int chunk) {
    const DevInfo di = dev_info();
    const int per_sm = chunk == 128 ? blocks_per_sm(ahla_tc_smem(), 288, 2, di)
                                    : blocks_per_sm(ahla_chunk_smem(d, chunk), ahla_chunk_threads(d), 4, di);
    return make_plan(B, H, n, d, d, chunk, di.sms, per_sm);
}

static int ahla_pass(const AhlaArgs& a, int d, int chunk, bool summary, cudaStream_t st) {
    if (chunk == 128) return launch_ahla_tc(a, summary, reinterpret_cast<int*>(a.ws), st);
    return launch_ahla_chunk(a, d, chunk, summary, st);
}

size_t hla2_ahla_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize) {
    if (ahla_check(B, H, n, d, dv, chunk, dtype, normalize) != HLA2_OK) return (size_t)-1;
    const Plan p = ahla_plan(B, H, n, d, chunk);
    size_t bytes = p.nseg > 0 ? ahla_layout(p).total * sizeof(float) : 0;
    if (chunk == 128) {  // a call with a final state (which the query does not see) runs at width 64
        const Plan p64 = ahla_plan(B, H, n, d, 64);
        const size_t b64 = p64.nseg > 0 ? ahla_layout(p64).total * sizeof(float) : 0;
        bytes = b64 > bytes ? b64 : bytes;
    }
    return bytes;
}

int hla2_ahla_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n, int d, int dv,
                      const float* gamma, int normalize, int chunk, hla2_stream_t stream, const hla2_opts* opts) {
    NvtxScope nvtx("hla2_ahla_forward");
    if (!opts) return fail(HLA2_ERR_INVALID_ARG, "opts must not be NULL");
    int rc = ahla_check(B, H, n, d, dv, chunk, opts->dtype, normalize);
    if (rc != HLA2_OK) return rc;
    if (normalize && !isfinite(opts->eps)) return fail(HLA2_ERR_INVALID_ARG, "eps must be finite");
    if (opts->flags) return fail(HLA2_ERR_INVALID_ARG, "unknown flags for hla2_ahla_forward");
    const bool want_final = opts->final_state != nullptr;
    if (opts->init_state && !aligned16(opts->init_state))
        return fail(HLA2_ERR_INVALID_ARG, "init_state must be 16-byte aligned");
    // the tcgen05 kernel keeps no final state: such calls run at width 64 (the result does not
    // depend on the width; the workspace query covers both widths)
    if (want_final && chunk == 128) chunk = 64;
    if (want_final && !aligned16(opts->final_state))
        return fail(HLA2_ERR_INVALID_ARG, "final_state must be 16-byte aligned");
    const long BH = (long)B * H;
    if (BH == 0) return succeed();
    if (n == 0) {  // no tokens: the final state is the initial one (or the empty state)
        const size_t bytes = BH * ahla_state_floats(d, dv) * sizeof(float);
        cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream);
        if (want_final && (opts->init_state ? cudaMemcpyAsync(opts->final_state, opts->init_state, bytes,
                                                              cudaMemcpyDeviceToDevice, s0)
                                            : cudaMemsetAsync(opts->final_state, 0, bytes, s0)) != cudaSuccess)
            return cuda_fail("final state");
        return succeed();
    }
    if (!q || !k || !v || !out) return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must not be NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return fail(HLA2_ERR_INVALID_ARG, "q, k, v, out must be 16-byte aligned");
    const Plan p = ahla_plan(B, H, n, d, chunk);
    const AhlaLayout L = ahla_layout(p);
    const size_t need = L.total * sizeof(float);
    if (!opts->workspace || opts->workspace_bytes < need)
        return fail(HLA2_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", need,
                    opts->workspace ? opts->workspace_bytes : (size_t)0);
    if (!aligned16(opts->workspace)) return fail(HLA2_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    AhlaArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.BH = (int)BH;
    a.H = H;
    a.n = n;
    a.W = chunk;
    a.nchunks = p.nchunks;
    a.seg_chunks = p.seg_chunks;
    a.nseg = p.nseg;
    a.nsum = p.nseg - 1;
    a.gamma = gamma;
    a.normalize = normalize;
    a.eps = opts->eps;
    a.ws = static_cast<float*>(opts->workspace);
    a.L = L;
    a.final_state = opts->final_state;
    a.init_state = opts->init_state;
    const bool den_terms = normalize || want_final;  // m, n carried
    auto mark = [&](int i) {
        nvtx.phase(kPhaseNames[i]);
        if (opts->phase_events && i < opts->n_phase_events && opts->phase_events[i] &&
            cudaEventRecord(static_cast<cudaEvent_t>(opts->phase_events[i]), st) != cudaSuccess)
            cudaGetLastError();
    };
    cudaGetLastError();
    mark(0);
    if (launch_ahla_init(a, d, st)) return cuda_fail("AHLA carry-in initialisation");
    mark(1);
    // chunk 128 (tcgen05) with more than one segment: the summary pass also stores the
    // segment-local Inner in out, over every segment, and the output pass starts from it
    const bool stored_inner = chunk == 128 && p.nseg > 1;
    if (p.nseg > 1) {
        const int steps = p.nseg - 1, seg_tokens = p.seg_chunks * chunk;
        const size_t dd = (size_t)d * d;
        AhlaArgs b = a;
        b.seg0 = 0;
        b.nseg_launch = stored_inner ? p.nseg : steps;
        b.store_inner = stored_inner ? 1 : 0;
        if (ahla_pass(b, d, chunk, true, st)) return cuda_fail("AHLA segment summaries");
        mark(2);
        if (launch_linear_scan(a.ws + L.PB, a.ws + L.Pin, a.BH, H, steps, dd, a.nsum * dd, p.nseg * dd, true, gamma,
                               seg_tokens, 1, st) ||
            (den_terms && launch_linear_scan(a.ws + L.mB, a.ws + L.min, a.BH, H, steps, d, a.nsum * (size_t)d,
                                             p.nseg * (size_t)d, true, gamma, seg_tokens, 1, st)) ||
            launch_ahla_cross(a, d, st) ||
            launch_linear_scan(a.ws + L.EB, a.ws + L.Ein, a.BH, H, steps, dd, a.nsum * dd, p.nseg * dd, true, gamma,
                               seg_tokens, 1, st) ||
            (den_terms && launch_linear_scan(a.ws + L.nB, a.ws + L.nin, a.BH, H, steps, d, a.nsum * (size_t)d,
                                             p.nseg * (size_t)d, true, gamma, seg_tokens, 1, st)))
            return cuda_fail("AHLA segment scan");
    } else {
        mark(2);
    }
    mark(3);
    AhlaArgs o = a;
    o.seg0 = 0;
    o.nseg_launch = p.nseg;
    if (stored_inner ? launch_ahla_tc_out_i(o, reinterpret_cast<int*>(a.ws), st) : ahla_pass(o, d, chunk, false, st))
        return cuda_fail("AHLA output pass");
    mark(4);
    mark(5);
    return succeed();
}

static int state_convert(const float* src, float* dst, int N, int H, int d, int dv, hla2_stream_t stream,
                         bool to_compact) {
    if (N < 0 || H < 0) return fail(HLA2_ERR_INVALID_ARG, "N, H must be >= 0 (got %d, %d)", N, H);
    if (!dim_ok(d) || !dim_ok(dv))
        return fail(HLA2_ERR_INVALID_ARG, "d and dv must be 16, 32, 64 or 128 (got %d, %d)", d, dv);
    const long heads = (long)N * H;
    if (heads == 0) return succeed();
    if (!src || !dst) return fail(HLA2_ERR_INVALID_ARG, "state pointers must not be NULL");
    const size_t nsrc = heads * (to_compact ? raw_state_floats(d, dv) : compact_state_floats(d, dv));
    const size_t ndst = heads * (to_compact ? compact_state_floats(d, dv) : raw_state_floats(d, dv));
    if (src < dst + ndst && dst < src + nsrc) return fail(HLA2_ERR_INVALID_ARG, "source and destination overlap");
    cudaGetLastError();
    if (launch_state_compact(src, dst, heads, d, dv, to_compact, reinterpret_cast<cudaStream_t>(stream)))
        return cuda_fail("state layout conversion");
    return succeed();
}

int hla2_state_to_compact(const float* state, float* compact, int N, int H, int d, int dv, hla2_stream_t stream) {
    return state_convert(state, compact, N, H, d, dv, stream, true);
}

int hla2_state_from_compact(const float* compact, float* state, int N, int H, int d, int dv,
                            hla2_stream_t stream) {
    return state_convert(compact, state, N, H, d, dv, stream, false);
}

}  // extern "C"
