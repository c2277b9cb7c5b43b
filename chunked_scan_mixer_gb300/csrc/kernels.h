// Internal interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace hla2 {

// Workspace of the AHLA forward (float offsets, d == dv): segment summaries P_B, E_B
// (d x dv), R_B (d x d), m_B, n_B (d); carries P_in, E_in, m_in, n_in per segment start.
struct AhlaLayout {
    size_t PB, EB, RB, mB, nB, Pin, Ein, min, nin, total;
};
inline AhlaLayout ahla_layout(const Plan& p) {
    AhlaLayout L;
    const size_t BH = p.BH, ns = p.nseg, nsm = p.nseg > 1 ? p.nseg - 1 : 0;
    const size_t dd = (size_t)p.d * p.d, d = p.d;
    size_t o = kStatusFloats;
    L.PB = o;  o = align64(o + BH * nsm * dd);
    L.EB = o;  o = align64(o + BH * nsm * dd);
    L.RB = o;  o = align64(o + BH * nsm * dd);
    L.mB = o;  o = align64(o + BH * nsm * d);
    L.nB = o;  o = align64(o + BH * nsm * d);
    L.Pin = o; o = align64(o + BH * ns * dd);
    L.Ein = o; o = align64(o + BH * ns * dd);
    L.min = o; o = align64(o + BH * ns * d);
    L.nin = o; o = align64(o + BH * ns * d);
    L.total = o;
    return L;
}

// AHLA streaming state of one head: P d*dv | E d*dv | m d | n d.
__host__ __device__ inline size_t ahla_state_floats(int d, int dv) { return 2 * (size_t)d * dv + 2 * (size_t)d; }

// Arguments of one AHLA chunk-kernel launch.
struct AhlaArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int BH, H, n, W, nchunks, seg_chunks, nseg, seg0, nseg_launch, nsum;
    const float* gamma;
    int normalize;
    float eps;
    float* ws;
    AhlaLayout L;
    float* final_state;  // nullable: [BH][2 d dv + 2 d] = P | E | m | n after token n
                         // (first-order mode of the tcgen05 kernel: [BH][d*dv] = P only)
    const float* init_state;  // nullable: the same layout, the state before token 0
    // tcgen05 summary pass (chunk 128): also store the segment-local Inner (the first-order
    // output with the value moment accumulated from the segment start, bf16) in out, for the
    // output pass launch_ahla_tc_out_i; the launch then covers every segment.
    int store_inner;
};
int launch_ahla_chunk(const AhlaArgs& a, int d, int W, bool summary, cudaStream_t st);
int launch_ahla_init(const AhlaArgs& a, int d, cudaStream_t st);
int launch_ahla_cross(const AhlaArgs& a, int d, cudaStream_t st);
size_t ahla_chunk_smem(int d, int W);
int ahla_chunk_threads(int d);
// tcgen05 AHLA chunk kernel (d = dv = 64, chunk 128, unnormalised; ahla_tc.cu)
bool ahla_tc_available();
size_t ahla_tc_smem();
// first_order: the pass computes masked first-order linear attention (out = Inner; the
// summaries keep only P_B), the inner pass of the third-order output.
int launch_ahla_tc(const AhlaArgs& a, bool summary, int* status, cudaStream_t st, bool first_order = false);
// Output pass from the stored segment-local Inner (tcgen05, chunk 128): only E is carried
// from chunk to chunk.
int launch_ahla_tc_out_i(const AhlaArgs& a, int* status, cudaStream_t st);

// Arguments of one chunk-kernel launch (summary or output pass of the forward).
struct ChunkArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int BH, H, n;
    int W;            // chunk width
    int nchunks, seg_chunks, nseg;
    int seg0;         // first segment of this launch (blockIdx.x + seg0)
    int nseg_launch;  // segments in this launch (grid.x)
    int nsum;         // segment summaries stored per head (nseg - 1, or nseg)
    const float* gamma;
    int normalize;
    float eps;
    int want_final;
    float* ws;        // forward workspace (floats)
    FwdLayout L;
    bf16* chunk_states;  // state-export pass: bf16 (S | Z) at every chunk start, [BH][nchunks][d*d + d*dv]
    // fp32 state-export pass of the SIMT kernel: (S | Z) at every chunk start,
    // [BH][nchunks][d*d + d*dv]; out may then be NULL.
    float* chunk_states_f32;
    // 1: unmasked output q^T S C (and denominator q^T S m).  The Z and y slots of the
    // summaries, the carries and the raw final state then hold C and m, which decay by
    // g per token, and no cross term enters the inter-segment scan.
    int unmasked;
};

// Chunk-kernel passes.
// tcgen05 kernel only: kSummaryP is the summary pass that also stores the segment-local
// p_t = S_t q_t (bf16, key moment accumulated from zero at the segment start) in `out`, over
// every segment; kOutputP is the output pass that starts from it.
enum ChunkMode { kSummary = 0, kOutput = 1, kStates = 2, kOutStates = 3, kOutputP = 4, kSummaryP = 5 };

// Arguments of the reverse-mode chunk kernel (bf16, d == dv).
struct BwdArgs {
    const bf16* q;
    const bf16* k;
    const bf16* v;
    const bf16* dout;
    bf16* dq;
    bf16* dk;
    bf16* dv;
    int BH, H, n, W, nchunks, seg_chunks, nseg;
    const float* gamma;
    float* ws;
    size_t ZhB, ShB;           // reverse summaries, float offsets, [BH][nseg][...]
    size_t Zh_end, Sh_end;     // reverse carries at segment ends, [BH][nseg][...]
    const bf16* chunk_states;  // forward (S | Z) bf16 at every chunk start
};

// Arguments of the fp32 reverse-mode chunk kernel (SIMT, any d, dv; bwd_chunk_simt.cu).
struct BwdArgsF {
    const float* q;
    const float* k;
    const float* v;
    const float* dout;
    float* dq;
    float* dk;
    float* dv;
    int BH, H, n, W, nchunks, seg_chunks, nseg;
    const float* gamma;
    float* ws;
    size_t ZhB, ShB;             // reverse summaries, float offsets, [BH][nseg][...]
    size_t Zh_end, Sh_end;       // reverse carries at segment ends, [BH][nseg][...]; updated in place
    const float* chunk_states;   // forward (S | Z) fp32 at every chunk start
};
// Resident CTAs per SM of the SIMT chunk kernels as their registers allow (their launch
// bounds): two of the forward kernel, one of the reverse-mode kernel.
constexpr int kSimtFwdCtas = 2, kSimtBwdCtas = 1;
int launch_bwd_chunk_simt(const BwdArgsF& a, int d, int dv, bool rsum, cudaStream_t st);
size_t bwd_chunk_simt_smem(int d, int dv, int W);

// Reverse-mode chunk kernel: rsum = true stores each segment's reverse summary,
// false writes dq, dk, dv.  d == dv in {16,32,64,128}; W in {16,32,64} (32 max for d = 128).
int launch_bwd_chunk_mma(const BwdArgs& a, int d, int W, bool rsum, cudaStream_t st);
size_t bwd_chunk_mma_smem(int d, int W);  // 0 if not compiled

// Reverse decayed suffix scan over segments (segment lengths from n, W, seg_chunks):
//   dst[nseg-1] = 0;  dst[s-1] = g^(power L_s) dst[s] + src[s]
int launch_reverse_scan(const float* src, float* dst, int BH, int H, int nseg, size_t E,
                        const float* gamma, int n, int W, int seg_chunks, int power, cudaStream_t st);
// In place: ShB[s] += g^(L_s) Zh_end[s] C_B[s]^T for s >= 1.
int launch_reverse_cross(const BwdArgs& b, const float* CB, int d, int dv, cudaStream_t st);

// ratio-normalised backward: quotient-rule glue (bwd_normalize.cu)
// [v | 1 | 0 ...] (w columns) from v (dv columns, bf16 or float32)
int launch_widen_values(const void* v, float* ve, size_t rows, int dv, int w, bool is_bf16, cudaStream_t st);
// [dL/dnum | dL/dden | 0 ...] from dout (dv columns) and [num | den | .] (w columns)
int launch_quotient_rule(const void* dout, const float* nd, float* dnd, size_t rows, int dv, int w, float eps,
                         bool is_bf16, cudaStream_t st);
// the first dv columns of [dv | .] (w columns), as bf16 or float32
int launch_narrow_values(const float* dve, void* out, size_t rows, int dv, int w, bool is_bf16, cudaStream_t st);
int launch_convert_bf16_f32(const bf16* src, float* dst, size_t count, cudaStream_t st);  // count % 8 == 0
int launch_convert_f32_bf16(const float* src, bf16* dst, size_t count, cudaStream_t st);

// Tensor-core (mma.sync bf16) chunk kernel: d == dv in {16,32,64,128}, W in {16,32,64,128}.
// Returns 0 on success, -1 on a CUDA error, -2 if the shape is not compiled.  With
// a.unmasked only the kSummary and kOutput modes exist and track_cm is ignored.
int launch_fwd_chunk_mma(const ChunkArgs& a, int d, int dv, int W, int mode, bool track_cm,
                         cudaStream_t st);
size_t fwd_chunk_mma_smem(int d, int dv, int W, bool track_cm);  // 0 if not compiled

// tcgen05 chunk kernel (bf16, d = dv = 64, chunk 128, unnormalised, modes kSummary and
// kOutput).  status: int word in the workspace set on a wait timeout.  Returns 0, -1 (CUDA
// error) or -2 (tensor maps unavailable).
bool fwd_chunk_tc_available();
size_t fwd_chunk_tc_smem();
int launch_fwd_chunk_tc(const ChunkArgs& a, int mode, int* status, cudaStream_t st);

// SIMT fp32-arithmetic chunk kernel, any d, dv <= 128 (multiples of 8), W <= 128;
// inputs float32 (is_bf16 = false) or bf16.
int launch_fwd_chunk_simt(const ChunkArgs& a, int d, int dv, int W, bool summary, bool track_cm,
                          bool is_bf16, cudaStream_t st);
size_t fwd_chunk_simt_smem(int d, int dv, int W, bool track_cm);

// Inter-segment scan and state conversion kernels (float32).
int launch_init_carry(const ChunkArgs& a, int d, int dv, const float* init_state, cudaStream_t st);
// One job of launch_linear_scans: a decayed prefix as launch_linear_scan computes it.
struct ScanJob {
    const float* src;
    float* dst;
    size_t E, src_hs, dst_hs;
    int store_all, power;
};
constexpr int kMaxScanJobs = 3;
struct ScanJobs {
    ScanJob job[kMaxScanJobs];
    int blocks[kMaxScanJobs];
    int n;
};
// Up to kMaxScanJobs independent scans over the same heads and steps in one launch.
int launch_linear_scans(const ScanJob* jobs, int njobs, int BH, int H, int nsteps, const float* gamma,
                        int step_tokens, cudaStream_t st);
int launch_linear_scan(const float* src, float* dst, int BH, int H, int nsteps, size_t E,
                       size_t src_head_stride, size_t dst_head_stride, bool store_all,
                       const float* gamma, int step_tokens, int power, cudaStream_t st);
int launch_cross(const ChunkArgs& a, int d, int dv, bool with_y, cudaStream_t st);
// Final state on the stored-p path (bf16, d = dv = 64): every segment's query and p moments
// (m_B, y_B, from q and the p stored in out), then the carry into the last segment combined with
// its summary and converted to the packed public state (final_state).
int launch_seg_moments64(const ChunkArgs& a, cudaStream_t st);
int launch_final_combine64(const ChunkArgs& a, float* final_state, cudaStream_t st);
int launch_finalize(const ChunkArgs& a, int d, int dv, float* final_state, cudaStream_t st);

// Decode step.
int launch_decode_step(float* state, const void* q, const void* k, const void* v, void* out,
                       int N, int H, int d, int dv, const float* gamma, int normalize, float eps,
                       bool is_bf16, bool compact, bool unmasked, cudaStream_t st);
// Multi-query decode: key_state [N*Hk][d*d], head_state [N*Hk*group][2 d dv + 2 d] (C | G | m | h);
// q [N*Hk*group][d], k [N*Hk][d], v [N*Hk][dv]; gamma NULL or [Hk]; 1 <= group <= 8.
int launch_decode_mq(float* key_state, float* head_state, const void* q, const void* k, const void* v, void* out,
                     int N, int Hk, int group, int d, int dv, const float* gamma, int normalize, float eps,
                     bool is_bf16, bool unmasked, cudaStream_t st);
// Third-order streaming step (gamma = 1): state [heads][d*d + 2 d dv + 2 d] = S | P | Y | m | y.
int launch_hla3_decode_step(float* state, const void* q, const void* k, const void* v, void* out, long heads, int d,
                            int dv, int normalize, float eps, bool is_bf16, cudaStream_t st);
int launch_ahla_decode_step(float* state, const void* q, const void* k, const void* v, void* out, int N, int H,
                            int d, int dv, const float* gamma, int normalize, float eps, bool is_bf16,
                            cudaStream_t st);
// AHLA reverse mode (ahla_bwd.cu, SIMT float32, d == dv).  Workspace float offsets, each block
// [BH][nseg][d*d] (states: [BH][nchunks][2 d*d], P then E at every chunk start).
struct AhlaBwdLayout {
    size_t PB, EB, RB, Pin, Ein, EhB, PhB, Eh_end, Ph_end, states, total;
};
AhlaBwdLayout ahla_bwd_layout(int BH, int nseg, int nchunks, int d);
struct AhlaBwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    int BH, H, n, d, W, nchunks, seg_chunks, nseg;
    const float* gamma;
    float* ws;
    size_t PB, EB, RB, Pin, Ein, EhB, PhB, Eh_end, Ph_end, states;
};
int launch_ahla_backward(const AhlaBwdArgs& a, bool is_bf16, cudaStream_t st);
size_t ahla_bwd_smem(int d, int W);

// Masked first-order linear attention u_t = sum_{l <= t} g^(t-l) (q_t . k_l) v_l, the inner
// pass of the third-order output (linattn.cu).  Workspace floats: PB [BH][nseg-1][d*dv],
// Pin [BH][nseg][d*dv].
struct LaArgs {
    const void* q;
    const void* k;
    const void* v;
    void* u;
    int BH, H, n, d, dv, W, nchunks, seg_chunks, nseg, seg0;
    const float* gamma;
    float* ws;
    size_t PB, Pin;
    float* final_P;  // nullable: [BH][d*dv], the state P after the last token
};
int launch_first_order_forward(const LaArgs& a, bool is_bf16, cudaStream_t st);
// Third-order streaming state [S | P | Y | m | y] from the passes' final states: the
// second-order packed states (S, C, G, m, h) on values u (dv wide) and u1 (w wide), and the
// first-order final P for v (dv wide) and for the unit values (w wide, column 0 = key mass).
int launch_hla3_assemble_state(float* fin, const float* pk_num, const float* pk_den, const float* p_num,
                               const float* p_den, long heads, int d, int dv, int w, cudaStream_t st);
size_t first_order_smem(int d, int dv, int W);
// rows x w with column 0 = 1, in the input type (bf16 or float32)
int launch_unit_rows(void* e0, size_t rows, int w, bool is_bf16, cudaStream_t st);
// out[row][:] /= (den[row * w] + eps), in place, bf16 or float32
int launch_divide_rows(void* out, const void* den, size_t rows, int dv, int w, float eps, bool is_bf16,
                       cudaStream_t st);

// tcgen05 first-order chunked scan, d = dv = 128, chunk 128 (fo_tc.cu): the building block of
// the d = 128 training path.  One launch runs every segment of every head ([BH] x [nseg] CTAs).
struct FoArgs {
    int BH, H, n, nchunks, seg_chunks, nseg;
    const float* gamma;   // per head [H] (NULL: 1); the scan's decay is gamma^pow
    int pow, pow_next;    // decay powers of the scan and of its next summary
    const float* carry;   // [BH][nseg][128*128] carry into each segment (NULL: zero)
    int carry_mode;       // 0 as stored, 1 transposed, 2 symmetrised (carry + carry^T)
    float* summary;       // [BH][nseg][128*128] segment summaries written (summary launch / next summary)
    int* status;          // bounded-wait status word
    const float* carry2;  // the second pair's carry (launch_fo64_tc_out2; NULL: zero)
    int carry_mode2;      // as carry_mode, for carry2
};
bool fo_tc_available();
size_t fo_tc_max_smem();
// carry[bh][0][0 .. E) = 0 for every head of a [BH][nseg][E] array (and *status = 0)
int launch_fo_zero_first(float* carry, int BH, int nseg, int E, int* status, cudaStream_t st);
// summary[s] = sum_{i in s} g^(distance to the segment's end (forward) / start (reverse)) k_i v_i^T
int launch_fo_tc_summary(const FoArgs& a, const void* k, const void* v, bool reverse, cudaStream_t st);
// The final state's summaries in one pass over (q, p, v), d = dv = 128, per segment:
// summary = sum_i w_i q_i v_i^T, zsum = sum_i w_i^2 p_i v_i^T, msum = sum_i w_i q_i,
// ysum = sum_i w_i^2 p_i ([BH][nseg][128] for the moments), w_i = g^(distance to the segment's end).
int launch_fo_tc_summary_final(const FoArgs& a, const void* q, const void* p, const void* v, float* zsum,
                               float* msum, float* ysum, cudaStream_t st);
// out = (R)LA(x, k, v) with the carry (v == NULL: the values are the keys); r2 adds the swapped
// pair (v, k); next_sum 1 / 2 also writes the next summary over (out, the values) / (out, xv);
// add != NULL adds that partial.
int launch_fo_tc_out(const FoArgs& a, const void* x, const void* k, const void* v, bool r2, int next_sum,
                     const void* xv, const void* add, void* out, bool reverse, cudaStream_t st);
// Final state of the first-order-scan forward (d = dv = 128).  Per segment s of head bh the
// moments mB[bh][s] = sum_t g^(L-1-t) q_t and yB[bh][s] = sum_t g^(2(L-1-t)) p_t (p the full p,
// t the token's place in the segment of L tokens) come from the summary pass
// (launch_fo_tc_summary_final).
struct FoFinal {
    const float *SB, *Sin, *ZB, *Zin, *CB;  // [BH][nseg][d][d]: summaries and carries (S, Z); C summaries
    const float *Cl, *ml, *yl;              // [BH][d][d], [BH][d]: carries of C, m, y into the last segment
    const float *mB, *yB;                   // [BH][nseg][d]
    int BH, H, n, d, nseg, seg_tokens;
    const float* gamma;
};
// The carry into the last segment combined with its summaries (rho = g^L, L its tokens),
//   S = rho S_in + S_B, C = rho C_in + C_B, m = rho m_in + m_B, Z = rho^2 Z_in + Z_B,
//   y = rho^2 y_in + y_B, written as the packed state (S, C, G = S C - Z, m, h = S m - y).
int launch_fo_final_state(const FoFinal& f, float* final_state, cudaStream_t st);
// The same two launches for d = dv = 64 (fo64_tc.cu; [BH][nseg][64*64] summaries and carries).
size_t fo64_tc_max_smem();
int launch_fo64_tc_summary(const FoArgs& a, const void* k, const void* v, bool reverse, cudaStream_t st);
// out = (R)LA(x, k, v) + (R)LA(x2, k2, v), d = dv = 64: two query / key pairs with the same values
// in one pass, as one scan of the stacked pairs ([x | x2] . [k | k2], a 128 x 64 state whose row
// halves carry a.carry (mode a.carry_mode) and a.carry2 (mode a.carry_mode2)).
int launch_fo64_tc_out2(const FoArgs& a, const void* x, const void* k, const void* x2, const void* k2, const void* v,
                        void* out, bool reverse, cudaStream_t st);
int launch_fo64_tc_out(const FoArgs& a, const void* x, const void* k, const void* v, bool r2, int next_sum,
                       const void* xv, const void* add, void* out, bool reverse, cudaStream_t st);

// Bounded-wait self-test: waits on an mbarrier nobody arrives at; records site 90 in *status.
int launch_wait_timeout_selftest(int* status, cudaStream_t st);
// Debug build: one failing bounds check (site 1) that guards no access.
int launch_debug_check_selftest(cudaStream_t st);
#ifdef HLA2_DEBUG
// Debug words of the files with bounds checks (HLA2_DEBUG_READER): the recorded site or 0;
// clear resets the word.
int dbg_read_fwd_simt(bool clear);
int dbg_read_decode(bool clear);
int dbg_read_fwd_mma_d16(bool clear);
int dbg_read_fwd_mma_d32(bool clear);
int dbg_read_fwd_mma_d64(bool clear);
int dbg_read_fwd_mma_d128(bool clear);
int dbg_read_bwd_mma_d16(bool clear);
int dbg_read_bwd_mma_d32(bool clear);
int dbg_read_bwd_mma_d64(bool clear);
int dbg_read_bwd_mma_d128(bool clear);
int dbg_read_bwd_simt(bool clear);
int dbg_read_scan(bool clear);
int dbg_read_fo_tc(bool clear);
int dbg_read_fo64_tc(bool clear);
int dbg_read_selftest(bool clear);
#endif
int launch_state_compact(const float* src, float* dst, long heads, int d, int dv, bool to_compact, cudaStream_t st);

}  // namespace hla2
