/*
 * hla2.h -- C ABI of the GB300 (sm_103a) library for masked second-order
 * Higher-order Linear Attention (HLA-2).
 *
 * What the library computes (page "Higher-order Linear Attention", technical summary,
 * item "1. Zweite Ordnung HLA"; section summary §2, §3.1, §4.3), per head and token t:
 *
 *   S_t = g S_{t-1} + k_t k_t^T          (key second moment,        d x d)
 *   C_t = g C_{t-1} + q_t v_t^T          (query-value accumulator,   d x dv)
 *   m_t = g m_{t-1} + q_t                (query mass,                d)
 *   G_t = g^2 G_{t-1} + g k_t (k_t^T C_{t-1})   (cross summary,      d x dv)
 *   h_t = g^2 h_{t-1} + g k_t (k_t^T m_{t-1})   (cross summary,      d)
 *   o_t = q_t^T (S_t C_t - G_t)                 (masked output,      dv)
 *   den_t = q_t^T (S_t m_t - h_t);  normalised output o_t / (den_t + eps)
 *
 * g is a fixed per-head decay in (0, 1] (1 = no decay).  Equivalently
 * o_t = sum_{i <= j <= t} g^((t-i)+(t-j)) (q_t . k_i)(k_i . q_j) v_j: the key index
 * never comes after the value index, and the pair i == j is kept.
 *
 * Conventions shared by every entry point
 *   - Every pointer is a DEVICE pointer unless stated otherwise; the caller owns every
 *     buffer.  The library allocates no device or host memory and keeps no state
 *     across calls except a thread-local error message.
 *   - Tensors are contiguous, head-major, row-vector layout:
 *       q, k [B, H, n, d];  v, out, dout [B, H, n, dv];  dq, dk [B, H, n, d];
 *       dv [B, H, n, dv].  Element type given by hla2_opts.dtype (HLA2_F32 or
 *       HLA2_BF16; every tensor of one call has the same type).
 *   - gamma: device float array [H], or NULL for no decay.  Values must lie in (0, 1];
 *     they are read on the device only and are not validated there.
 *   - Packed state of one head (decode layout), float32:
 *       [ S d*d (row-major) | C d*dv | G d*dv | m d | h d ]   (hla2_state_floats)
 *     init_state / final_state / the decode state are [B or N, H] such blocks.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).  The
 *     compute calls only enqueue work (no host synchronisation, no device allocation);
 *     hla2_forward and the decode steps can be captured in a CUDA graph.  Within one
 *     forward, a kernel may start its prologue while the previous kernel of the call
 *     drains (programmatic dependent launch); it waits for that kernel's results before
 *     touching memory.
 *     Return value: HLA2_OK or a negative error code; hla2_last_error() describes the
 *     last failure on the calling host thread.  Argument errors are detected on the
 *     host before anything is launched; launch errors map to HLA2_ERR_CUDA.
 *   - Supported sizes: d, dv in {16, 32, 64, 128}; chunk in {16, 32, 64, 128};
 *     any n >= 0 (the last chunk may be partial); B, H >= 0.  Pointers must be
 *     16-byte aligned.  A combination the kernels do not cover returns
 *     HLA2_ERR_UNSUPPORTED.  For hla2_forward (and its workspace and plan queries)
 *     chunk is the widest width used: where no kernel covers (dtype, d, dv) at that
 *     width, the call runs at the widest smaller one that has a kernel, since the output
 *     does not depend on the width (only the floating-point summation order does).
 */
#ifndef HLA2_H_
#define HLA2_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st* hla2_stream_t;

enum {
    HLA2_OK = 0,
    HLA2_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size, bad flag       */
    HLA2_ERR_UNSUPPORTED = -2, /* valid request outside the compiled kernel set      */
    HLA2_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required         */
    HLA2_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed        */
    HLA2_ERR_TIMEOUT = -5      /* reserved: a bounded device-side wait gave up       */
};

enum { HLA2_F32 = 0, HLA2_BF16 = 1 };

/* Options that trail the positional arguments.  Zero-initialise and set what you use. */
typedef struct {
    int dtype;              /* HLA2_F32 | HLA2_BF16: type of q, k, v, out, dout, grads      */
    float eps;              /* ratio-normalisation epsilon (used when normalize != 0)         */
    void* workspace;        /* device scratch of >= the size the *_workspace_bytes query gives */
    size_t workspace_bytes; /* its size in bytes                                              */
    const float* init_state;/* nullable: packed state [B, H] to continue from (forward only)  */
    float* final_state;     /* nullable: receives the packed state after token n (forward)   */
    /* Optional profiling hook: cudaEvent_t handles recorded on `stream` at phase
     * boundaries of hla2_forward: [0] start, [1] after the carry-in set-up, [2] after
     * the segment-summary pass, [3] after the inter-segment scan, [4] after the output
     * pass, [5] after the final-state conversion.  The first n_phase_events are used;
     * NULL / 0 records nothing.  The caller creates and owns the events. */
    void* const* phase_events;
    int n_phase_events;
    /* HLA2_FLAG_* bits; 0 for plain calls. */
    int flags;
} hla2_opts;

/*
 * hla2_opts.flags for a training step, forward then backward on the same inputs:
 *   HLA2_FLAG_SAVE_FOR_BACKWARD (hla2_forward): also keep in the workspace what the
 *     backward would otherwise recompute: the segment summaries and the bf16 (S, Z) at
 *     every chunk start, at the backward's chunk width.  The workspace must hold
 *     hla2_backward_workspace_bytes(B, H, n, d, dv, chunk, dtype) bytes.  Only for what
 *     hla2_backward covers: bf16, d == dv, normalize == 0, no init_state or final_state
 *     (else HLA2_ERR_UNSUPPORTED).
 *   HLA2_FLAG_STATES_SAVED (hla2_backward): the workspace holds those pieces from a
 *     SAVE_FOR_BACKWARD forward with the same q, k, gamma, sizes and chunk, untouched since;
 *     the backward then skips its forward recomputation.  The library cannot check that
 *     the workspace is still intact: passing this flag otherwise gives wrong gradients.
 * and for the unmasked output (hla2_forward, hla2_decode_step):
 *   HLA2_FLAG_UNMASKED: o_t = q_t^T S_t C_t, the bilinear form of the prefix moments without
 *     the G correction (section summary §3, "numerator-style bilinear form"), and with
 *     normalize the denominator q_t^T S_t m_t.  Every (key, value) pair up to t counts,
 *     weighted g^((t-i)+(t-j)); the chunk scan combines (S, C, m) by decayed addition (the
 *     unmasked monoid, section summary §4.1).  G and h are not tracked: a forward's
 *     final_state holds them as 0, init_state's are ignored, and the decode step leaves them
 *     untouched.  Not with HLA2_FLAG_SAVE_FOR_BACKWARD (HLA2_ERR_UNSUPPORTED): the backward
 *     covers the masked output.
 */
enum {
    HLA2_FLAG_SAVE_FOR_BACKWARD = 1,
    HLA2_FLAG_STATES_SAVED = 2,
    HLA2_FLAG_COMPACT_STATE = 4,
    HLA2_FLAG_UNMASKED = 8
};

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int hla2_version(void);

/* Message describing the last error returned on this host thread ("" if none). */
const char* hla2_last_error(void);

/* Floats in one packed head state: d*d + 2*d*dv + 2*d. */
size_t hla2_state_floats(int d, int dv);

/*
 * Scratch bytes hla2_forward needs for these arguments (0 is a valid answer).
 * Depends on the arguments and on the number of SMs of the current device.
 * Returns (size_t)-1 for arguments hla2_forward would reject.
 */
size_t hla2_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                    int normalize, int want_final_state);

/*
 * Strictly causal masked HLA-2 forward, chunk-parallel (section summary §4, §4.2, §5;
 * technical summary item "4. Paralleles Training durch assoziative Scans").
 * q, k, v -> out.  The sequence is cut into chunks of width `chunk`; chunks are
 * grouped into segments; per-segment summaries are combined by an exclusive scan
 * with the masked semidirect product (cross term S_B C_A) to give each segment
 * its carry-in; every token's output is then formed from its inclusive state.
 * normalize != 0 divides by the masked denominator (+ opts->eps); on the tcgen05 path (bf16,
 * d = dv = 64, chunk 128, masked) the denominator is formed in the output pass's epilogue.
 * bf16 at d = dv = 128, chunk 128, masked and unnormalised without init_state runs on the
 * tcgen05 first-order scans, with or without final_state.
 * opts must be non-NULL (dtype and workspace).  init_state continues a previous
 * sequence; final_state receives the state after the last token (prefill for
 * hla2_decode_step).  opts->flags may hold HLA2_FLAG_SAVE_FOR_BACKWARD or
 * HLA2_FLAG_UNMASKED (the unmasked output, with the same workspace size).
 * out must not overlap q, k or v: on the masked bf16 path at d = dv = 64, chunk 128 with
 * more than one segment, a final state or normalize != 0, the summary pass first stores
 * p_t = S_t q_t (the key moment accumulated from the segment start) in out, and the output
 * pass overwrites it.
 */
int hla2_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n,
                 int d, int dv, const float* gamma, int normalize, int chunk,
                 hla2_stream_t stream, const hla2_opts* opts);

/*
 * The segmentation hla2_forward will use for these arguments on the current device:
 * *nseg segments of *seg_chunks chunks per head, and *launches kernel launches per
 * call (normalize and want_final_state as passed to hla2_forward).  Any output pointer
 * may be NULL.  Returns HLA2_OK, HLA2_ERR_INVALID_ARG, or HLA2_ERR_UNSUPPORTED where no
 * kernel covers the sizes at any width <= chunk (as hla2_forward).  The segmentation is the same
 * with HLA2_FLAG_UNMASKED; the launch count is the masked output's (the unmasked one
 * needs fewer).
 */
int hla2_forward_plan(int B, int H, int n, int d, int dv, int chunk, int dtype, int normalize,
                      int want_final_state, int* nseg, int* seg_chunks, int* launches);

/*
 * Reads the status word at the start of a workspace used by hla2_forward / hla2_backward:
 * HLA2_OK, or HLA2_ERR_TIMEOUT when a bounded device-side wait of a kernel gave up (the
 * kernel then drained and returned; its outputs are not valid).  The word is cleared by
 * the next call that uses the workspace.  Synchronises `stream`.
 */
int hla2_workspace_status(const void* workspace, hla2_stream_t stream);

/*
 * Self-test of the bounded device-side waits: launches one CTA that waits, with the same
 * bounded poll the tcgen05 kernels use (over a second), on an mbarrier that nothing
 * arrives at.  The wait gives up, records site 90 in the status word at the start of
 * `workspace` (>= 16 bytes, 16-byte aligned) and the kernel returns; hla2_workspace_status
 * then reports HLA2_ERR_TIMEOUT, and the context stays usable.  Asynchronous on `stream`.
 */
int hla2_selftest_wait_timeout(void* workspace, hla2_stream_t stream);

/*
 * Debug build (the library compiled with HLA2_DEBUG, as `python -m chunked_scan_mixer_gb300.build
 * --debug` makes it in chunked_scan_mixer_gb300/_build_debug/): the kernels of the float32 and
 * mma.sync chunk paths, the forward and backward inter-segment scans, the decode steps and the
 * tcgen05 first-order scans check the indices of their global-memory accesses against the
 * buffers' extents.  A failed check records a site code (positive) in a device word, skips
 * the access and lets the kernel finish: nothing traps.
 * hla2_debug_status synchronises the device and returns the first recorded site, 0 when every
 * check passed since the last clear (clear != 0 resets the words), or HLA2_ERR_UNSUPPORTED in
 * the normal build.  hla2_debug_selftest launches one kernel whose only check fails without
 * guarding any access, so that hla2_debug_status then reports site 1 (HLA2_ERR_UNSUPPORTED in
 * the normal build).
 */
int hla2_debug_status(int clear);
int hla2_debug_selftest(hla2_stream_t stream);

/* Scratch bytes hla2_backward needs; (size_t)-1 for rejected arguments. */
size_t hla2_backward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                     int normalize);

/*
 * Reverse-mode chunk scan (section summary §4.2: gradients equal to those of the
 * serial recurrence): given dout = dL/dout, writes dq, dk, dv.  bf16 tensors with d == dv
 * run on the tensor-core kernels (chunk width <= 64, <= 32 at d = 128); float32 tensors of
 * any d, dv on SIMT float32 kernels (chunk width <= 32).
 * normalize == 0: gradients of the unnormalised output.  normalize == 1: gradients of
 * o / (den + opts->eps) by the quotient rule (section summary §5.1).  num and den are the
 * unnormalised outputs for the values v and for the value rows (1, 0, ..., 0), so the call
 * runs one unnormalised backward with the widened values [v | 1 | 0 ...] (dv + 16 columns):
 * its forward part gives [num | den], the upstream gradient is
 * [dout / (den + eps) | -(dout . num) / (den + eps)^2 | 0 ...], and its reverse part gives dq,
 * dk and [dv | .].  dq and dk are then the sum of a numerator part and a denominator part that
 * can each be tens of times larger than the sum, so this composition always runs in float32
 * (bf16 tensors are widened first and the gradients rounded at the end; any d, dv); the
 * workspace then also holds those float32 intermediates.  init_state and final_state in opts must be NULL
 * (gradients start from the empty state); HLA2_FLAG_STATES_SAVED needs bf16 and
 * normalize == 0.
 */
int hla2_backward(const void* q, const void* k, const void* v, const void* dout, void* dq,
                  void* dk, void* dv_out, int B, int H, int n, int d, int dv,
                  const float* gamma, int normalize, int chunk, hla2_stream_t stream,
                  const hla2_opts* opts);

/*
 * One streaming decode step for N*H independent heads (section summary §3.1: online
 * updates at O(d^2 + d dv) per token, constant state).  state [N, H] packed float32
 * blocks, updated in place; q, k [N, H, d]; v, out [N, H, dv].  The cross summaries
 * G, h are advanced from the pre-update C, m; the output uses the updated state.
 * opts may be NULL (then dtype = HLA2_BF16, eps = 1e-6); no workspace is used.
 * opts->flags may hold HLA2_FLAG_COMPACT_STATE and HLA2_FLAG_UNMASKED (then G and h are
 * neither read nor written).
 */
int hla2_decode_step(float* state, const void* q, const void* k, const void* v, void* out,
                     int N, int H, int d, int dv, const float* gamma, int normalize,
                     hla2_stream_t stream, const hla2_opts* opts);

/*
 * AHLA reverse mode (section summary §4.2's reverse-mode scan applied to the AHLA
 * recurrence): given dout = dL/dout of the unnormalised hla2_ahla_forward output, writes dq,
 * dk, dv.  float32 or bf16 tensors [B, H, n, d], d == dv.  bf16 with d = dv = 64 and
 * chunk >= 128: tcgen05 first-order chunked scans at width 128 (the output is two chained
 * first-order scans with the same queries and keys, u = LA(q, k, v) and o = LA(q, k, u), and
 * its gradients six more, dk and dq each two with the same values run as one pass; fp32 state,
 * bf16 u and du between the passes).  Otherwise float32
 * arithmetic on SIMT kernels at a chunk width <= min(chunk, 32): the passes recompute the
 * forward (segment summaries P_B, E_B, R_B, the forward scan, the state at every chunk start)
 * and then run the reverse summaries, the reverse scan (cross term rho R_B^T Eh_end) and the
 * gradient pass.  normalize must be 0; no flags, init_state or final_state.  Tensor pointers
 * must be 16-byte aligned.  Workspace: hla2_ahla_backward_workspace_bytes.
 */
size_t hla2_ahla_backward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                          int normalize);
int hla2_ahla_backward(const void* q, const void* k, const void* v, const void* dout, void* dq, void* dk,
                       void* dv_out, int B, int H, int n, int d, int dv, const float* gamma, int normalize,
                       int chunk, hla2_stream_t stream, const hla2_opts* opts);

/*
 * Masked third-order HLA at gamma = 1 (technical summary item "3. Dritte Ordnung HLA": the
 * product A A^T A with A = Q K^T, masked so that strict causality holds; section summary:
 * the chunk scan of this case is exact for gamma = 1).  Every factor and the partial product
 * of the first two carry the causal mask:
 *   o_t = sum_{j <= t} sum_{i <= j} sum_{l <= j} (q_t . k_i)(k_i . q_j)(q_j . k_l) v_l,
 * i.e. the masked second-order output whose values are the first-order outputs
 * u_j = sum_{l <= j} (q_j . k_l) v_l.  It runs as a chunked first-order pass into the
 * workspace (the tcgen05 AHLA kernel in a first-order mode for bf16, d = dv = 64; SIMT
 * otherwise), then hla2_forward on (q, k, u) -- the tcgen05 kernels for bf16, d = dv = 64,
 * chunk 128.  normalize != 0 divides by the same sum with v -> 1 (+ opts->eps), computed the
 * same way with the value rows (1, 0, ..., 0).  gamma must be NULL (HLA2_ERR_UNSUPPORTED
 * otherwise); no init_state; opts->final_state receives the streaming state after token n
 * in the layout of hla2_hla3_decode_step (prefill; the unit-value passes then run as for
 * normalize); opts->flags must be 0.  Tensors as for hla2_forward; the workspace is
 * hla2_hla3_forward_workspace_bytes.
 */
size_t hla2_hla3_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                         int normalize, int want_final_state);
int hla2_hla3_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n, int d,
                      int dv, const float* gamma, int normalize, int chunk, hla2_stream_t stream,
                      const hla2_opts* opts);

/*
 * Third-order streaming step (gamma = 1; the masked streaming of technical summary item 3,
 * under the reading of hla2_hla3_forward).  state [N, H] float32 blocks of
 * hla2_state_floats(d, dv) floats laid out [S^K d*d | P^KV d*dv | Y d*dv | m^K d | y d],
 * updated in place: S^K += k k^T, P^KV += k v^T, m^K += k; with p = S^K q and u = P^KV^T q,
 * Y += p u^T and y += p (q . m^K); out = q^T Y (normalize: / (q^T y + opts->eps)).
 * q, k [N, H, d]; v, out [N, H, dv].  A zero state is the empty prefix.  opts may be NULL
 * (dtype bf16, eps 1e-6); opts->flags must be 0.
 */
int hla2_hla3_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H,
                          int d, int dv, int normalize, hla2_stream_t stream, const hla2_opts* opts);

/* Floats in one head's part of the multi-query state: C d*dv | G d*dv | m d | h d. */
size_t hla2_mq_head_state_floats(int d, int dv);

/*
 * Decode step with multi-query sharing of the key moment (section summary §5.2: sharing
 * cuts the state from O(h d^2) to O(d^2 + h d dv)).  The `group` query heads of each key
 * group share the token's key and value, hence one S per group; C, G, m, h stay per head.
 * key_state [N, Hk] blocks of S (d*d float32, packed), head_state [N, Hk*group] blocks of
 * hla2_mq_head_state_floats(d, dv) float32 -- both updated in place; q [N, Hk*group, d]
 * (the heads of key group j are j*group .. j*group+group-1); k [N, Hk, d]; v [N, Hk, dv];
 * out [N, Hk*group, dv]; gamma NULL or [Hk] (one decay per group, since S carries it).
 * 1 <= group <= 8.  The result equals hla2_decode_step on heads whose k and v are the
 * group's and whose S blocks are the group's S.  opts may be NULL; opts->flags may hold
 * HLA2_FLAG_UNMASKED; HLA2_FLAG_COMPACT_STATE gives HLA2_ERR_UNSUPPORTED.  One CTA per
 * query head; the CTAs of a key group form a cluster that streams the group's S once (a
 * block of rows each) and shares u = S' q through distributed shared memory; no workspace.
 */
int hla2_decode_step_mq(float* key_state, float* head_state, const void* q, const void* k, const void* v,
                        void* out, int N, int Hk, int group, int d, int dv, const float* gamma, int normalize,
                        hla2_stream_t stream, const hla2_opts* opts);

/*
 * Asymmetric HLA (AHLA, technical summary item "2. Asymmetrische Lineare Aufmerksamkeit
 * hoeherer Ordnung"; section summary §6): the masked left-cascaded product
 * Q (K^T Q)(K^T V),
 *   o_t = sum_{j <= t} sum_{i <= j} g^(t-i) (q_t . k_j)(q_j . k_i) v_i,
 * streamed with P_t = g P + k v^T, E_t = g E + k (q^T P_t), o_t = q_t^T E_t (and m, n for
 * the denominator with v -> 1; normalised output o / (den + eps)).  Chunk-parallel over an
 * exclusive scan of segment summaries (P, E, m, n, R = sum k q^T) (section summary §6.2).
 * bf16 q, k, v, out [B, H, n, d], d == dv in {16, 32, 64, 128}, chunk 32 or 64 (legacy
 * tensor cores), or chunk 128 for d = dv = 64 unnormalised (tcgen05).
 * opts->final_state receives the AHLA state after token n, [B, H] blocks of
 * hla2_ahla_state_floats = [P d*dv | E d*dv | m d | n d] (a call at chunk 128 with a final
 * state runs at width 64: the tcgen05 kernel keeps none); opts->init_state (any chunk) in the
 * same layout continues from that state; opts->flags must be 0.
 * Workspace as for hla2_forward; a timed-out device-side wait of the tcgen05 kernel is
 * reported by hla2_workspace_status.
 */
size_t hla2_ahla_forward_workspace_bytes(int B, int H, int n, int d, int dv, int chunk, int dtype,
                                         int normalize);
int hla2_ahla_forward(const void* q, const void* k, const void* v, void* out, int B, int H, int n,
                      int d, int dv, const float* gamma, int normalize, int chunk,
                      hla2_stream_t stream, const hla2_opts* opts);

/* Floats in one head's AHLA state: 2*d*dv + 2*d. */
size_t hla2_ahla_state_floats(int d, int dv);

/*
 * One AHLA streaming step for N*H heads (section summary §6.1: O(d dv) per token):
 * state [N, H] blocks [P | E | m | n] float32 updated in place; q, k [N, H, d]; v, out
 * [N, H, dv].  P, m are advanced first, the inner read q^T P uses the updated P, then E, n,
 * and the output q^T E reads the updated E.  opts may be NULL (dtype HLA2_BF16, eps 1e-6).
 */
int hla2_ahla_decode_step(float* state, const void* q, const void* k, const void* v, void* out,
                          int N, int H, int d, int dv, const float* gamma, int normalize,
                          hla2_stream_t stream, const hla2_opts* opts);

/*
 * Compact decode state.  S is symmetric (a sum of decayed k k^T), so a head's state can
 * keep only its upper block triangle: row a holds S[a][b] for b = 4*floor(a/4) .. d-1,
 * rows back to back (d*(d+4)/2 floats; every row starts on 16 bytes), followed by C, G, m,
 * h as in the packed layout.  hla2_decode_step with opts->flags & HLA2_FLAG_COMPACT_STATE
 * reads and writes states in this layout, moving 16 % fewer bytes per step at
 * d = dv = 128.  The same bit is an argument error for every other entry point.
 */
size_t hla2_compact_state_floats(int d, int dv);

/*
 * Convert N*H head states between the packed and the compact layouts (device pointers,
 * asynchronous on stream, src and dst must not overlap).  To compact: S's upper block
 * triangle is kept (a packed S that is not exactly symmetric loses its other triangle);
 * from compact: S is mirrored.  Returns HLA2_OK, HLA2_ERR_INVALID_ARG or HLA2_ERR_CUDA.
 */
int hla2_state_to_compact(const float* state, float* compact, int N, int H, int d, int dv,
                          hla2_stream_t stream);
int hla2_state_from_compact(const float* compact, float* state, int N, int H, int d, int dv,
                            hla2_stream_t stream);

/*
 * hla2_forward for callers that cannot allocate device memory (no counterpart in the
 * paper: it exists for the library's users).  Some callers have no way to provide the
 * scratch workspace that hla2_forward needs: plug-in hosts that hand a kernel only its
 * input and output buffers, or programs with no device allocator of their own.  This entry point
 * takes the same tensors and flags as hla2_forward (dtype and eps given directly; no
 * initial or final state) and allocates nothing: its scratch is a fixed 32 MiB array in
 * the library's device memory, present on every GPU on which the library's kernels are
 * loaded and held until the process exits.
 *   - Sizes whose workspace (hla2_forward_workspace_bytes) exceeds 32 MiB are rejected
 *     with HLA2_ERR_WORKSPACE and a message; use hla2_forward with a workspace for them.
 *   - The first call on a device looks up the array's device address for that device.
 *   - All calls on a device share the array, which keeps the last call's contents (nothing
 *     in it needs to start at zero).  Calls whose executions overlap on the GPU (different
 *     streams, or graphs running concurrently) race on it and give wrong results:
 *     serialise them.
 */
int hla2_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H, int n,
                         int d, int dv, const float* gamma, int normalize, int chunk, int dtype,
                         float eps, hla2_stream_t stream);

/*
 * The status word of the allocation-free entry point's scratch array on the current device
 * (no counterpart in the paper either).  Its kernels report a bounded device-side wait that
 * gave up in the first word of their scratch, as hla2_forward does in its workspace; the
 * caller of hla2_forward_noalloc has no address for that array, so this reads it:
 * HLA2_OK, or HLA2_ERR_TIMEOUT when a wait of the last hla2_forward_noalloc call on this
 * device gave up (its output is then not valid).  The next call clears the word, so read
 * it after a call and before the next one.  Synchronises `stream`.
 */
int hla2_noalloc_status(hla2_stream_t stream);

/*
 * hla2_selftest_wait_timeout run on the allocation-free entry point's scratch array: a
 * wait that nothing ends gives up and records site 90 there, after which
 * hla2_noalloc_status reports HLA2_ERR_TIMEOUT until the next hla2_forward_noalloc call.
 * Asynchronous on `stream`; no fault, and the context stays usable.
 */
int hla2_noalloc_selftest_wait_timeout(hla2_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HLA2_H_ */
