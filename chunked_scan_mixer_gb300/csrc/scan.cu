// Inter-segment scan of the masked HLA-2 forward (float32).
//
// Segment summaries (S_B, C_B, Z_B, m_B, y_B) of consecutive segments A (earlier)
// and B combine with the masked semidirect product (page "Higher-order Linear
// Attention", section summary §4.2, §4.3; technical summary item "4. Paralleles
// Training durch assoziative Scans", cross term S^K_B C^QV_A).  In the (S, C, m, Z, y)
// coordinates used on the GPU (Z = S C - G, y = S m - h) the combine with
// rho = g^len(B) reads
//     S = rho S_A + S_B,   C = rho C_A + C_B,   m = rho m_A + m_B,
//     Z = rho^2 Z_A + Z_B + rho S_A C_B,   y = rho^2 y_A + y_B + rho S_A m_B,
// (the pairs with key in A and value in B are kept by the mask).  The exclusive scan
// over segments therefore splits into
//   1. a decayed prefix sum of S (elementwise, linear_scan_kernel),
//   2. independent products X_s = Z_B[s] + rho S_in[s] C_B[s] (cross_kernel),
//   3. a decayed (rho^2) prefix sum of X (linear_scan_kernel again).
#include "kernels.h"
#include "simt_tile.cuh"

namespace hla2 {

namespace {

constexpr int kThreads = 256;

// Carry into segment 0 from the optional packed initial state (S, C, G, m, h):
// Z0 = S0 C0 - G0 and y0 = S0 m0 - h0; zero without an initial state.  The unmasked
// output carries C0 and m0 in those slots and ignores G0 and h0.
__global__ void __launch_bounds__(kThreads)
    init_carry_kernel(const ChunkArgs a, int D, int DV, const float* init) {
    pdl_trigger();  // the summary pass may start its prologue (it waits before touching memory)
    const int bh = blockIdx.x, tid = threadIdx.x;
    if (bh == 0 && tid == 0) *reinterpret_cast<int*>(a.ws) = 0;  // clear the status word
    const size_t s0 = (size_t)bh * a.nseg;  // segment 0 of this head
    float* Sin = a.ws + a.L.Sin + s0 * D * D;
    float* Zin = a.ws + a.L.Zin + s0 * D * DV;
    float* yin = a.ws + a.L.yin + s0 * D;
    float* Cl = a.ws + a.L.Clast + (size_t)bh * D * DV;
    float* ml = a.ws + a.L.mlast + (size_t)bh * D;
    if (!init) {
        for (int i = tid; i < D * D; i += kThreads) Sin[i] = 0.f;
        for (int i = tid; i < D * DV; i += kThreads) Zin[i] = Cl[i] = 0.f;
        for (int i = tid; i < D; i += kThreads) yin[i] = ml[i] = 0.f;
        return;
    }
    const PackOff po = pack_off(D, DV);
    const float* st = init + (size_t)bh * (size_t)raw_state_floats(D, DV);
    const float *S0 = st + po.S, *C0 = st + po.C, *G0 = st + po.G, *m0 = st + po.m, *h0 = st + po.h;
    for (int i = tid; i < D * D; i += kThreads) Sin[i] = S0[i];
    if (a.unmasked) {
        for (int i = tid; i < D * DV; i += kThreads) Zin[i] = Cl[i] = C0[i];
        for (int i = tid; i < D; i += kThreads) yin[i] = ml[i] = m0[i];
        return;
    }
    for (int i = tid; i < D * DV; i += kThreads) {
        const int r = i / DV, c = i % DV;
        float s = 0.f;
        for (int x = 0; x < D; ++x) s += S0[r * D + x] * C0[x * DV + c];
        Zin[i] = s - G0[i];
        Cl[i] = C0[i];
    }
    for (int r = tid; r < D; r += kThreads) {
        float s = 0.f;
        for (int x = 0; x < D; ++x) s += S0[r * D + x] * m0[x];
        yin[r] = s - h0[r];
        ml[r] = m0[r];
    }
}

// Decayed prefix over segments, one thread per element:
//   acc_0 = dst[head][0][e];  acc_{s+1} = rho_h^power acc_s + src[head][s][e]
// with rho_h = g_h^step_tokens.  store_all writes every acc_s (s >= 1) to
// dst[head][s][e]; otherwise only the last one to dst[head][0][e].
__global__ void __launch_bounds__(kThreads)
    linear_scan_kernel(const float* __restrict__ src, float* __restrict__ dst, int BH, int H,
                       int nsteps, size_t E, size_t src_hs, size_t dst_hs, int store_all,
                       const float* gamma, int step_tokens, int power) {
    pdl_trigger();
    pdl_wait();
    const size_t gid = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (gid >= (size_t)BH * E) return;
    const int bh = (int)(gid / E);
    const size_t e = gid % E;
    const float rho = pow_decay(log2f(head_decay(gamma, bh, H)), (float)step_tokens * (float)power);
    const float* s = src + (size_t)bh * src_hs + e;
    float* d = dst + (size_t)bh * dst_hs + e;
    // every access below stays in head bh's part of src and dst (debug build: checked once)
    if (!HLA2_IN(e < E && (size_t)nsteps * E <= src_hs && (size_t)(store_all ? nsteps : 0) * E < dst_hs, 701)) return;
    float acc = d[0];
    constexpr int U = 8;
    int t = 0;
    for (; t + U <= nsteps; t += U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = s[(size_t)(t + u) * E];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc = rho * acc + x[u];
            if (store_all) d[(size_t)(t + u + 1) * E] = acc;
        }
    }
    for (; t < nsteps; ++t) {
        acc = rho * acc + s[(size_t)t * E];
        if (store_all) d[(size_t)(t + 1) * E] = acc;
    }
    if (!store_all) d[0] = acc;
}

// Up to kMaxScanJobs independent linear scans (each as linear_scan_kernel) in one launch:
// blocks [b_j, b_j + blocks_j) serve job j.
__global__ void __launch_bounds__(kThreads)
    linear_scans_kernel(const ScanJobs jobs, int BH, int H, int nsteps, const float* gamma, int step_tokens) {
    pdl_trigger();
    pdl_wait();
    int j = 0, b = blockIdx.x;
    while (j + 1 < jobs.n && b >= jobs.blocks[j]) b -= jobs.blocks[j++];
    const ScanJob& J = jobs.job[j];
    const size_t E = J.E;
    const size_t gid = (size_t)b * kThreads + threadIdx.x;
    if (gid >= (size_t)BH * E) return;
    const int bh = (int)(gid / E);
    const size_t e = gid % E;
    const float rho = pow_decay(log2f(head_decay(gamma, bh, H)), (float)step_tokens * (float)J.power);
    const float* src = J.src + (size_t)bh * J.src_hs + e;
    float* dst = J.dst + (size_t)bh * J.dst_hs + e;
    if (!HLA2_IN(e < E && (size_t)nsteps * E <= J.src_hs && (size_t)(J.store_all ? nsteps : 0) * E < J.dst_hs, 703))
        return;
    float acc = dst[0];
    constexpr int U = 8;
    int t = 0;
    for (; t + U <= nsteps; t += U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = src[(size_t)(t + u) * E];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc = rho * acc + x[u];
            if (J.store_all) dst[(size_t)(t + u + 1) * E] = acc;
        }
    }
    for (; t < nsteps; ++t) {
        acc = rho * acc + src[(size_t)t * E];
        if (J.store_all) dst[(size_t)(t + 1) * E] = acc;
    }
    if (!J.store_all) dst[0] = acc;
}

// Copy n floats (n a multiple of 4, both pointers 16-byte aligned) from global to shared
// memory: every load of a thread is issued before its first store, so that the L2 round
// trips overlap.
template <int N>
__device__ __forceinline__ void copy_to_smem(float* dst, const float* __restrict__ src, int tid) {
    static_assert(N % 4 == 0, "float4 copies");
    constexpr int N4 = N / 4, IT = (N4 + kThreads - 1) / kThreads;
    float4 r[IT];
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int i = tid + k * kThreads;
        if (i < N4) r[k] = reinterpret_cast<const float4*>(src)[i];
    }
#pragma unroll
    for (int k = 0; k < IT; ++k) {
        const int i = tid + k * kThreads;
        if (i < N4) reinterpret_cast<float4*>(dst)[i] = r[k];
    }
}

// X_s = Z_B[s] + rho S_in[s] C_B[s] (and, with WITH_Y, Xy_s = y_B[s] + rho S_in[s] m_B[s]),
// in place.  256 threads in a 16 x 16 grid; thread (tr, tc) computes rows tr + 16 i and the
// TN consecutive columns TN tc .. of X in fp32 from shared-memory copies of S_in[s], C_B[s].
template <int TM, int TN, bool WITH_Y>
__global__ void __launch_bounds__(kThreads) cross_kernel(const ChunkArgs a, int seg_tokens) {
    constexpr int D = 16 * TM, DV = 16 * TN;
    extern __shared__ __align__(16) float sm[];
    float* Ss = sm;            // D x D
    float* Cs = Ss + D * D;    // D x DV
    float* ms = Cs + D * DV;   // D
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const size_t sb = (size_t)bh * a.nsum + s;        // summary index
    const size_t si = (size_t)bh * a.nseg + s;        // carry index
    const float* Sin = a.ws + a.L.Sin + si * D * D;
    const float* CB = a.ws + a.L.CB + sb * D * DV;
    float* ZB = a.ws + a.L.ZB + sb * D * DV;
    copy_to_smem<D * D>(Ss, Sin, tid);
    copy_to_smem<D * DV>(Cs, CB, tid);
    if (WITH_Y)
        for (int i = tid; i < D; i += kThreads) ms[i] = a.ws[a.L.mB + sb * D + i];
    const int tr = tid / 16, tc0 = (tid % 16) * TN;
    // this thread's part of Z_B, loaded while the copies land
    float zb[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) zb[i][j] = ZB[(size_t)(tr + 16 * i) * DV + tc0 + j];
    __syncthreads();
    const float rho = pow_decay(log2f(head_decay(a.gamma, bh, a.H)), (float)seg_tokens);
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int x = 0; x < D; ++x) {
        float av[TM], bv[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) av[i] = Ss[(tr + 16 * i) * D + x];
#pragma unroll
        for (int j = 0; j < TN; ++j) bv[j] = Cs[x * DV + tc0 + j];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] += av[i] * bv[j];
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) ZB[(size_t)(tr + 16 * i) * DV + tc0 + j] = zb[i][j] + rho * acc[i][j];
    if (WITH_Y) {
        float* yB = a.ws + a.L.yB + sb * D;
        for (int r = tid; r < D; r += kThreads) {
            float t = 0.f;
            for (int x = 0; x < D; ++x) t += Ss[r * D + x] * ms[x];
            yB[r] += rho * t;
        }
    }
}

// Query and p moments of every kept segment summary for the final state and the normalised
// output of the stored-p path (d = 64, bf16):
//   m_B[s] = sum_t g^(L-1-t) q_t,   y_B[s] = sum_t g^(2(L-1-t)) p^sl_t,
// t the token's place in segment s of L tokens, p^sl the segment-local p that the summary pass
// stored in out (read here before the output pass replaces it).  The tcgen05 summary pass
// forms S_B, C_B and Z_B but not these two vectors.  The unmasked output carries m in the y
// slot, so there y_B = m_B and p is not read.  One CTA per (segment, head, half of the
// features); thread (row, j) sums features 32 z + 8j .. +7 over tokens row, row + 64, ...
__global__ void __launch_bounds__(kThreads) seg_moments64_kernel(const ChunkArgs a) {
    constexpr int D = 64, HALF = 32, ROWS = kThreads / 4;
    __shared__ float red_m[ROWS][HALF + 1], red_y[ROWS][HALF + 1];
    pdl_trigger();
    pdl_wait();
    const int s = blockIdx.x, bh = blockIdx.y, z = blockIdx.z, tid = threadIdx.x;
    const int row = tid / 4, j = tid % 4;
    const int t0 = s * a.seg_chunks * a.W, t1 = min(t0 + a.seg_chunks * a.W, a.n);
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    const int f0 = HALF * z + 8 * j;
    const bf16* q = static_cast<const bf16*>(a.q) + (size_t)bh * a.n * D + f0;
    const bf16* pp = static_cast<const bf16*>(a.out) + (size_t)bh * a.n * D + f0;
    float am[8], ay[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) am[u] = ay[u] = 0.f;
    constexpr int U = 4;  // tokens a thread has in flight (loads issued before use)
    for (int t = t0 + row; t < t1; t += ROWS * U) {
        uint4 qv[U], pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int tu = t + ROWS * u;
            if (tu < t1) {
                qv[u] = *reinterpret_cast<const uint4*>(q + (size_t)tu * D);
                if (!a.unmasked) pv[u] = *reinterpret_cast<const uint4*>(pp + (size_t)tu * D);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int tu = t + ROWS * u;
            if (tu < t1) {
                const float w = pow_decay(log2g, (float)(t1 - 1 - tu)), w2 = a.unmasked ? w : w * w;
                const uint32_t qw[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
                const uint32_t pw[4] = {a.unmasked ? qv[u].x : pv[u].x, a.unmasked ? qv[u].y : pv[u].y,
                                        a.unmasked ? qv[u].z : pv[u].z, a.unmasked ? qv[u].w : pv[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    am[2 * e] += w * __uint_as_float(qw[e] << 16);
                    am[2 * e + 1] += w * __uint_as_float(qw[e] & 0xFFFF0000u);
                    ay[2 * e] += w2 * __uint_as_float(pw[e] << 16);
                    ay[2 * e + 1] += w2 * __uint_as_float(pw[e] & 0xFFFF0000u);
                }
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        red_m[row][8 * j + u] = am[u];
        red_y[row][8 * j + u] = ay[u];
    }
    __syncthreads();
    if (tid < 2 * HALF) {
        const int f = tid % HALF;
        float (*red)[HALF + 1] = tid < HALF ? red_m : red_y;
        float acc = 0.f;
        for (int r = 0; r < ROWS; ++r) acc += red[r][f];
        const size_t sb = (size_t)bh * a.nsum + s;
        a.ws[(tid < HALF ? a.L.mB : a.L.yB) + sb * D + HALF * z + f] = acc;
    }
}

// Final state of the stored-p path (d = dv = 64): the carry into the last segment combined with
// that segment's summary by the masked combine (rho = g^L of the last segment; the unmasked
// output adds S, C and m without cross terms),
//   S = rho S_in + S_B,  C = rho C_in + C_B,  m = rho m_in + m_B,
//   Z = rho^2 Z_in + Z_B + rho S_in C_B,  y = rho^2 y_in + y_B + rho S_in m_B,
// then G = S C - Z and h = S m - y, written as the packed public state.  Four CTAs a head, CTA
// rb forming rows 16 rb .. 16 rb + 15 of every part; the products run from shared-memory
// copies (its 16 rows of S_in, then of S, and all of C_B, then of C), thread (r, c) forming
// row r and columns 4c .. 4c + 3.
__global__ void __launch_bounds__(kThreads) final_combine64_kernel(const ChunkArgs a, float* final_state) {
    constexpr int D = 64, RB = 16;
    __shared__ __align__(16) float Ss[RB * D];
    __shared__ __align__(16) float Cs[D * D];
    __shared__ float ms[D], ys[RB];
    pdl_trigger();
    pdl_wait();
    const int rb = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int r0 = RB * rb;
    const int last = a.nseg - 1;
    const int L = a.n - last * a.seg_chunks * a.W;
    const float rho = pow_decay(log2f(head_decay(a.gamma, bh, a.H)), (float)L), rho2 = rho * rho;
    const size_t ci = (size_t)bh * a.nseg + last, sb = (size_t)bh * a.nsum + last;
    const float* Sin = a.ws + a.L.Sin + ci * D * D;
    const float* Zin = a.ws + a.L.Zin + ci * D * D;
    const float* yin = a.ws + a.L.yin + ci * D;
    const float* Cin = a.ws + a.L.Clast + (size_t)bh * D * D;
    const float* min_ = a.ws + a.L.mlast + (size_t)bh * D;
    const float *SB = a.ws + a.L.SB + sb * D * D, *CB = a.ws + a.L.CB + sb * D * D, *ZB = a.ws + a.L.ZB + sb * D * D;
    const float *mB = a.ws + a.L.mB + sb * D, *yB = a.ws + a.L.yB + sb * D;
    float* o = final_state + (size_t)bh * raw_state_floats(D, D);
    const PackOff po = pack_off(D, D);
    if (a.unmasked) {
        // unmasked output: S, C (in the Z slots) and m (in the y slots) add up decayed, without
        // cross terms; G and h are not tracked and are written as 0
        for (int i = tid; i < RB * D; i += kThreads) {
            const size_t e = (size_t)r0 * D + i;
            o[po.S + e] = rho * Sin[e] + SB[e];
            o[po.C + e] = rho * Zin[e] + ZB[e];
            o[po.G + e] = 0.f;
        }
        for (int i = tid; i < RB; i += kThreads) {
            o[po.m + r0 + i] = rho * yin[r0 + i] + yB[r0 + i];
            o[po.h + r0 + i] = 0.f;
        }
        return;
    }
    const int r = tid / 16, c4 = (tid % 16) * 4;  // row r0 + r, columns c4 .. c4 + 3
    auto product = [&](float (&acc)[4]) {          // acc = (Ss Cs)[r][c4 ..]
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll 8
        for (int x = 0; x < D; ++x) {
            const float av = Ss[r * D + x];
            const float4 bv = *reinterpret_cast<const float4*>(&Cs[x * D + c4]);
            acc[0] += av * bv.x;
            acc[1] += av * bv.y;
            acc[2] += av * bv.z;
            acc[3] += av * bv.w;
        }
    };
    // every global read of this thread issued before the first use: S_in and S_B rows, C_B and
    // C_in (all rows), its Z_in and Z_B entries (float4 each)
    constexpr int NC = D * D / 4 / kThreads;  // float4 of C per thread
    static_assert(RB * D / 4 == kThreads && NC * 4 * kThreads == D * D, "one float4 of a row block per thread");
    auto ld4 = [](const float* p) { return *reinterpret_cast<const float4*>(p); };
    const float4 sin4 = ld4(Sin + (size_t)r0 * D + 4 * tid), sb4 = ld4(SB + (size_t)r0 * D + 4 * tid);
    const size_t ez = (size_t)(r0 + r) * D + c4;
    const float4 zin4 = ld4(Zin + ez), zb4 = ld4(ZB + ez);
    float4 cb4[NC], cin4[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        cb4[k] = ld4(CB + 4 * (tid + kThreads * k));
        cin4[k] = ld4(Cin + 4 * (tid + kThreads * k));
    }
    const float mb = tid < D ? mB[tid] : 0.f, mi = tid < D ? min_[tid] : 0.f;
    const float yi = tid < RB ? yin[r0 + tid] : 0.f, yb = tid < RB ? yB[r0 + tid] : 0.f;
    // Z and y rows from the carry S_in and the last summary's C_B, m_B
    *reinterpret_cast<float4*>(Ss + 4 * tid) = sin4;
#pragma unroll
    for (int k = 0; k < NC; ++k) *reinterpret_cast<float4*>(Cs + 4 * (tid + kThreads * k)) = cb4[k];
    if (tid < D) ms[tid] = mb;
    __syncthreads();
    float zt[4], acc[4];
    product(acc);
    zt[0] = rho2 * zin4.x + zb4.x + rho * acc[0];
    zt[1] = rho2 * zin4.y + zb4.y + rho * acc[1];
    zt[2] = rho2 * zin4.z + zb4.z + rho * acc[2];
    zt[3] = rho2 * zin4.w + zb4.w + rho * acc[3];
    if (tid < RB) {
        float t = 0.f;
        for (int x = 0; x < D; ++x) t += Ss[tid * D + x] * ms[x];
        ys[tid] = rho2 * yi + yb + rho * t;
    }
    __syncthreads();  // every product of S_in is done
    // S rows, all of C, and m after the last token (in place); this CTA writes its rows
    {
        const float4 sv = make_float4(rho * sin4.x + sb4.x, rho * sin4.y + sb4.y, rho * sin4.z + sb4.z,
                                      rho * sin4.w + sb4.w);
        *reinterpret_cast<float4*>(Ss + 4 * tid) = sv;
        *reinterpret_cast<float4*>(o + po.S + (size_t)r0 * D + 4 * tid) = sv;
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int e = 4 * (tid + kThreads * k);
        const float4 cv = make_float4(rho * cin4[k].x + cb4[k].x, rho * cin4[k].y + cb4[k].y,
                                      rho * cin4[k].z + cb4[k].z, rho * cin4[k].w + cb4[k].w);
        *reinterpret_cast<float4*>(Cs + e) = cv;
        if (e >= r0 * D && e < (r0 + RB) * D) *reinterpret_cast<float4*>(o + po.C + e) = cv;
    }
    if (tid < D) {
        ms[tid] = rho * mi + mb;
        if (tid >= r0 && tid < r0 + RB) o[po.m + tid] = ms[tid];
    }
    __syncthreads();
    product(acc);  // G = S C - Z
#pragma unroll
    for (int u = 0; u < 4; ++u) o[po.G + ez + u] = acc[u] - zt[u];
    if (tid < RB) {  // h = S m - y
        float t = 0.f;
        for (int x = 0; x < D; ++x) t += Ss[tid * D + x] * ms[x];
        o[po.h + r0 + tid] = t - ys[tid];
    }
}

// Final state of the first-order-scan forward: CTA (rb, bh) forms rows 32 rb .. 32 rb + 31 of
// every part.  The combined C (all D rows) and the CTA's rows of S sit in shared memory; the
// rows of G = S C come from the register-tiled products of simt_tile.cuh.  Loads are float4 and
// issued together; with a single segment the carries into it are zero and are not read.
template <int D>
__global__ void __launch_bounds__(kThreads) fo_final_state_kernel(const FoFinal f, float* final_state) {
    constexpr int RB = 32, LDS = simt::pad(D), NC4 = D * D / 4 / kThreads, NS4 = RB * D / 4 / kThreads;
    static_assert(NC4 * 4 * kThreads == D * D && NS4 * 4 * kThreads == RB * D, "whole float4 per thread");
    extern __shared__ __align__(16) float fsm[];
    float* Cs = fsm;                // [D][D]
    float* Ss = Cs + D * D;         // [RB][LDS]
    float* ms = Ss + RB * LDS;      // [D]
    float* ys = ms + D;             // [RB]
    pdl_trigger();
    pdl_wait();
    const int rb = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int r0 = RB * rb, last = f.nseg - 1;
    const bool carry = f.nseg > 1;
    const int L = f.n - last * f.seg_tokens;
    const float rho = pow_decay(log2f(head_decay(f.gamma, bh, f.H)), (float)L), rho2 = rho * rho;
    const size_t si = (size_t)bh * f.nseg + last, DD = (size_t)D * D;
    const float *SB = f.SB + si * DD, *Sin = f.Sin + si * DD, *ZB = f.ZB + si * DD, *Zin = f.Zin + si * DD;
    const float *CB = f.CB + si * DD, *Cl = f.Cl + (size_t)bh * DD;
    const float *mB = f.mB + si * D, *yB = f.yB + si * D, *ml = f.ml + (size_t)bh * D, *yl = f.yl + (size_t)bh * D;
    float* o = final_state + (size_t)bh * raw_state_floats(D, D);
    const PackOff po = pack_off(D, D);
    auto ld4 = [](const float* p) { return *reinterpret_cast<const float4*>(p); };
    auto comb = [](float r, float4 a, float4 b) {  // r a + b
        return make_float4(fmaf(r, a.x, b.x), fmaf(r, a.y, b.y), fmaf(r, a.z, b.z), fmaf(r, a.w, b.w));
    };
    {  // C = rho C_in + C_B, all rows; this CTA's rows to the state
        float4 c[NC4];
#pragma unroll
        for (int k = 0; k < NC4; ++k) c[k] = ld4(CB + 4 * (tid + kThreads * k));
        if (carry)
#pragma unroll
            for (int k = 0; k < NC4; ++k) c[k] = comb(rho, ld4(Cl + 4 * (tid + kThreads * k)), c[k]);
#pragma unroll
        for (int k = 0; k < NC4; ++k) {
            const int e = 4 * (tid + kThreads * k);
            *reinterpret_cast<float4*>(Cs + e) = c[k];
            if (e >= r0 * D && e < (r0 + RB) * D) *reinterpret_cast<float4*>(o + po.C + e) = c[k];
        }
    }
    {  // S = rho S_in + S_B, this CTA's rows
        float4 sv[NS4];
#pragma unroll
        for (int k = 0; k < NS4; ++k) sv[k] = ld4(SB + (size_t)r0 * D + 4 * (tid + kThreads * k));
        if (carry)
#pragma unroll
            for (int k = 0; k < NS4; ++k) sv[k] = comb(rho, ld4(Sin + (size_t)r0 * D + 4 * (tid + kThreads * k)), sv[k]);
#pragma unroll
        for (int k = 0; k < NS4; ++k) {
            const int e = 4 * (tid + kThreads * k), r = e / D, c = e - r * D;
            *reinterpret_cast<float4*>(Ss + r * LDS + c) = sv[k];
            *reinterpret_cast<float4*>(o + po.S + (size_t)r0 * D + e) = sv[k];
        }
    }
    for (int i = tid; i < D; i += kThreads) {
        ms[i] = carry ? fmaf(rho, ml[i], mB[i]) : mB[i];
        if (i >= r0 && i < r0 + RB) o[po.m + i] = ms[i];
    }
    for (int i = tid; i < RB; i += kThreads) ys[i] = carry ? fmaf(rho2, yl[r0 + i], yB[r0 + i]) : yB[r0 + i];
    __syncthreads();
    // G = S C - (rho^2 Z_in + Z_B), this CTA's rows
    simt::with_rm(RB, D, [&](auto t) {
        constexpr int RM = decltype(t)::value;
        simt::for_blocks<RM>(RB, D, [&](int m0, int n0) {
            simt::Acc<RM> acc;
            simt::zero(acc);
            simt::mac_r<RM>(acc, Ss + m0 * LDS, LDS, Cs + n0, D, D);
#pragma unroll
            for (int i = 0; i < RM; ++i) {
                const size_t e = (size_t)(r0 + m0 + i) * D + n0;
                float4 z = ld4(ZB + e);
                if (carry) z = comb(rho2, ld4(Zin + e), z);
                const float g[4] = {acc[i][0] - z.x, acc[i][1] - z.y, acc[i][2] - z.z, acc[i][3] - z.w};
                simt::st4(o + po.G + e, g);
            }
        });
    });
    if (tid < RB) {  // h = S m - y
        float t = 0.f;
        for (int x = 0; x < D; ++x) t = fmaf(Ss[tid * LDS + x], ms[x], t);
        o[po.h + r0 + tid] = t - ys[tid];
    }
}

// Raw final (S, C, m, Z, y) -> packed public state (S, C, G = S C - Z, m, h = S m - y).
__global__ void __launch_bounds__(kThreads)
    finalize_kernel(const ChunkArgs a, int D, int DV, float* final_state) {
    const int bh = blockIdx.x, tid = threadIdx.x;
    const RawOff ro = raw_off(D, DV);
    const PackOff po = pack_off(D, DV);
    const float* r = a.ws + a.L.fin + (size_t)bh * raw_state_floats(D, DV);
    float* o = final_state + (size_t)bh * raw_state_floats(D, DV);
    const float *S = r + ro.S, *C = r + ro.C, *m = r + ro.m, *Z = r + ro.Z, *y = r + ro.y;
    for (int i = tid; i < D * D; i += kThreads) o[po.S + i] = S[i];
    if (a.unmasked) {  // C and m sit in the Z and y slots; G and h are not tracked
        for (int i = tid; i < D * DV; i += kThreads) {
            o[po.C + i] = Z[i];
            o[po.G + i] = 0.f;
        }
        for (int x = tid; x < D; x += kThreads) {
            o[po.m + x] = y[x];
            o[po.h + x] = 0.f;
        }
        return;
    }
    for (int i = tid; i < D * DV; i += kThreads) {
        const int x = i / DV, c = i % DV;
        float acc = 0.f;
        for (int j = 0; j < D; ++j) acc += S[x * D + j] * C[j * DV + c];
        o[po.C + i] = C[i];
        o[po.G + i] = acc - Z[i];
    }
    for (int x = tid; x < D; x += kThreads) {
        float acc = 0.f;
        for (int j = 0; j < D; ++j) acc += S[x * D + j] * m[j];
        o[po.m + x] = m[x];
        o[po.h + x] = acc - y[x];
    }
}

int finish_launch() { return cudaPeekAtLastError() == cudaSuccess ? 0 : -1; }

}  // namespace

int launch_init_carry(const ChunkArgs& a, int d, int dv, const float* init_state, cudaStream_t st) {
    if (a.BH <= 0) return 0;
    init_carry_kernel<<<a.BH, kThreads, 0, st>>>(a, d, dv, init_state);
    return finish_launch();
}

int launch_linear_scan(const float* src, float* dst, int BH, int H, int nsteps, size_t E,
                       size_t src_hs, size_t dst_hs, bool store_all, const float* gamma,
                       int step_tokens, int power, cudaStream_t st) {
    const size_t total = (size_t)BH * E;
    if (total == 0 || nsteps <= 0) return 0;
    const unsigned blocks = (unsigned)((total + kThreads - 1) / kThreads);
    if (launch_pdl(linear_scan_kernel, dim3(blocks), dim3(kThreads), 0, st, src, dst, BH, H, nsteps, E, src_hs,
                   dst_hs, store_all ? 1 : 0, gamma, step_tokens, power) != cudaSuccess)
        return -1;
    return finish_launch();
}

int launch_linear_scans(const ScanJob* jobs, int njobs, int BH, int H, int nsteps, const float* gamma,
                        int step_tokens, cudaStream_t st) {
    if (njobs <= 0 || njobs > kMaxScanJobs) return -1;
    if (BH <= 0 || nsteps <= 0) return 0;
    ScanJobs J{};
    unsigned total = 0;
    for (int i = 0; i < njobs; ++i) {
        J.job[i] = jobs[i];
        J.blocks[i] = (int)(((size_t)BH * jobs[i].E + kThreads - 1) / kThreads);
        total += (unsigned)J.blocks[i];
    }
    J.n = njobs;
    if (launch_pdl(linear_scans_kernel, dim3(total), dim3(kThreads), 0, st, J, BH, H, nsteps, gamma, step_tokens) !=
        cudaSuccess)
        return -1;
    return finish_launch();
}

template <int TM, int TN, bool WITH_Y>
int launch_cross_t(const ChunkArgs& a, cudaStream_t st) {
    constexpr int D = 16 * TM, DV = 16 * TN;
    const size_t smem = (size_t)(D * D + D * DV + D) * sizeof(float);
    if (cudaFuncSetAttribute(cross_kernel<TM, TN, WITH_Y>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    if (launch_pdl(cross_kernel<TM, TN, WITH_Y>, dim3(a.nseg - 1, a.BH), dim3(kThreads), smem, st, a,
                   a.seg_chunks * a.W) != cudaSuccess)
        return -1;
    return finish_launch();
}

// d in {16, 32, 64, 128}, dv in {16, 32, 48, 64, 80, 128, 144}; the largest (128 x 144) needs
// 137 KB of shared memory.
// with_y adds the denominator moment's cross term (needed by the normalised output and the
// final state only).
int launch_cross(const ChunkArgs& a, int d, int dv, bool with_y, cudaStream_t st) {
    if (a.nseg <= 1 || a.BH <= 0) return 0;
#define HLA2_CROSS(DD, VV)                                                                   \
    if (d == DD && dv == VV) {                                                               \
        constexpr int TM = DD / 16, TN = VV / 16;                                             \
        return with_y ? launch_cross_t<TM, TN, true>(a, st) : launch_cross_t<TM, TN, false>(a, st); \
    }
    HLA2_CROSS(16, 16) HLA2_CROSS(16, 32) HLA2_CROSS(16, 64) HLA2_CROSS(16, 128)
    HLA2_CROSS(32, 16) HLA2_CROSS(32, 32) HLA2_CROSS(32, 64) HLA2_CROSS(32, 128)
    HLA2_CROSS(64, 16) HLA2_CROSS(64, 32) HLA2_CROSS(64, 64) HLA2_CROSS(64, 128)
    HLA2_CROSS(128, 16) HLA2_CROSS(128, 32) HLA2_CROSS(128, 64) HLA2_CROSS(128, 128)
    // value widths dv + 16 of the normalised backward's widened values [v | e_0]
    HLA2_CROSS(16, 48) HLA2_CROSS(16, 80) HLA2_CROSS(16, 144)
    HLA2_CROSS(32, 48) HLA2_CROSS(32, 80) HLA2_CROSS(32, 144)
    HLA2_CROSS(64, 48) HLA2_CROSS(64, 80) HLA2_CROSS(64, 144)
    HLA2_CROSS(128, 48) HLA2_CROSS(128, 80) HLA2_CROSS(128, 144)
#undef HLA2_CROSS
    return -1;
}

int launch_seg_moments64(const ChunkArgs& a, cudaStream_t st) {
    if (a.nsum <= 0 || a.BH <= 0) return 0;  // the summaries kept: every segment but the last, or all
    if (launch_pdl(seg_moments64_kernel, dim3(a.nsum, a.BH, 2), dim3(kThreads), 0, st, a) != cudaSuccess) return -1;
    return finish_launch();
}

int launch_fo_final_state(const FoFinal& f, float* final_state, cudaStream_t st) {
    if (f.nseg <= 0 || f.BH <= 0) return 0;
    const size_t smem = ((size_t)f.d * f.d + 32 * (size_t)simt::pad(f.d) + f.d + 32) * sizeof(float);
    cudaError_t e;
    if (f.d == 128) {
        e = cudaFuncSetAttribute(fo_final_state_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = launch_pdl(fo_final_state_kernel<128>, dim3(f.d / 32, f.BH), dim3(kThreads), smem, st, f, final_state);
    } else if (f.d == 64) {
        e = cudaFuncSetAttribute(fo_final_state_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = launch_pdl(fo_final_state_kernel<64>, dim3(f.d / 32, f.BH), dim3(kThreads), smem, st, f, final_state);
    } else {
        e = cudaErrorInvalidValue;
    }
    return e == cudaSuccess ? finish_launch() : -1;
}

int launch_final_combine64(const ChunkArgs& a, float* final_state, cudaStream_t st) {
    if (a.nseg <= 0 || a.BH <= 0) return 0;
    if (launch_pdl(final_combine64_kernel, dim3(4, a.BH), dim3(kThreads), 0, st, a, final_state) != cudaSuccess)
        return -1;
    return finish_launch();
}

int launch_finalize(const ChunkArgs& a, int d, int dv, float* final_state, cudaStream_t st) {
    if (a.BH <= 0) return 0;
    finalize_kernel<<<a.BH, kThreads, 0, st>>>(a, d, dv, final_state);
    return finish_launch();
}

}  // namespace hla2

namespace hla2 {

namespace {

__device__ __forceinline__ int segment_tokens(int s, int n, int W, int seg_chunks) {
    const long start = (long)s * seg_chunks * W;
    const long len = (long)seg_chunks * W;
    return (int)(n - start < len ? n - start : len);
}

// Reverse decayed suffix over segments, one thread per element:
//   acc = 0 (nothing after the last segment); for s = nseg-1 .. 1:
//   acc = g^(power L_s) acc + src[s];  dst[s-1] = acc.   dst[nseg-1] = 0.
__global__ void __launch_bounds__(kThreads)
    reverse_scan_kernel(const float* __restrict__ src, float* __restrict__ dst, int BH, int H, int nseg,
                        size_t E, const float* gamma, int n, int W, int seg_chunks, int power) {
    pdl_trigger();
    pdl_wait();
    const size_t gid = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (gid >= (size_t)BH * E) return;
    const int bh = (int)(gid / E);
    const size_t e = gid % E;
    const float log2g = log2f(head_decay(gamma, bh, H));
    const float* s_ = src + (size_t)bh * nseg * E + e;
    float* d_ = dst + (size_t)bh * nseg * E + e;
    if (!HLA2_IN(e < E && nseg >= 1, 702)) return;
    float acc = 0.f;
    d_[(size_t)(nseg - 1) * E] = 0.f;
    constexpr int U = 8;  // steps s .. s - U + 1: their loads issued before the first use
    int s = nseg - 1;
    for (; s - U + 1 >= 1; s -= U) {
        float x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = s_[(size_t)(s - u) * E];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float rho = pow_decay(log2g, (float)power * (float)segment_tokens(s - u, n, W, seg_chunks));
            acc = rho * acc + x[u];
            d_[(size_t)(s - u - 1) * E] = acc;
        }
    }
    for (; s >= 1; --s) {
        const float rho = pow_decay(log2g, (float)power * (float)segment_tokens(s, n, W, seg_chunks));
        acc = rho * acc + s_[(size_t)s * E];
        d_[(size_t)(s - 1) * E] = acc;
    }
}

// ShB[s][f][a] += g^(L_s) sum_e Zh_end[s][f][e] C_B[s][a][e], for s >= 1: X = Zh C_B^T.
// 256 threads in a 16 x 16 grid; thread (tr, tc) computes rows tr + 16 i and the D/16
// consecutive columns of X from shared-memory copies of Zh_end[s] and C_B[s]^T (the latter
// stored with a row pitch of D + 1 floats).
template <int D, int DV>
__global__ void __launch_bounds__(kThreads) reverse_cross_kernel(const BwdArgs b, const float* CB) {
    constexpr int TM = D / 16, TN = D / 16, CP = D + 1;
    extern __shared__ __align__(16) float sm[];
    float* Zs = sm;            // D x DV
    float* Ct = sm + D * DV;   // DV x CP (transposed C_B)
    const int s = blockIdx.x + 1, bh = blockIdx.y, tid = threadIdx.x;
    const size_t si = (size_t)bh * b.nseg + s;
    const float* Zh = b.ws + b.Zh_end + si * D * DV;
    const float* C = CB + si * D * DV;
    float* Sh = b.ws + b.ShB + si * D * D;
    copy_to_smem<D * DV>(Zs, Zh, tid);
    {
        constexpr int N4 = D * DV / 4, IT = (N4 + kThreads - 1) / kThreads;
        float4 r[IT];
#pragma unroll
        for (int k = 0; k < IT; ++k) {
            const int i = tid + k * kThreads;
            if (i < N4) r[k] = reinterpret_cast<const float4*>(C)[i];
        }
#pragma unroll
        for (int k = 0; k < IT; ++k) {
            const int i = tid + k * kThreads;
            if (i < N4) {
                const int a = (4 * i) / DV, e = (4 * i) % DV;
                Ct[(e + 0) * CP + a] = r[k].x;
                Ct[(e + 1) * CP + a] = r[k].y;
                Ct[(e + 2) * CP + a] = r[k].z;
                Ct[(e + 3) * CP + a] = r[k].w;
            }
        }
    }
    const int tr = tid / 16, tc0 = (tid % 16) * TN;
    float sh[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) sh[i][j] = Sh[(size_t)(tr + 16 * i) * D + tc0 + j];
    __syncthreads();
    const float rho = pow_decay(log2f(head_decay(b.gamma, bh, b.H)), (float)segment_tokens(s, b.n, b.W, b.seg_chunks));
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int e = 0; e < DV; ++e) {
        float av[TM], bv[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) av[i] = Zs[(tr + 16 * i) * DV + e];
#pragma unroll
        for (int j = 0; j < TN; ++j) bv[j] = Ct[e * CP + tc0 + j];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] += av[i] * bv[j];
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) Sh[(size_t)(tr + 16 * i) * D + tc0 + j] = sh[i][j] + rho * acc[i][j];
}

template <int D, int DV>
int launch_reverse_cross_t(const BwdArgs& b, const float* CB, cudaStream_t st) {
    const size_t smem = ((size_t)D * DV + (size_t)DV * (D + 1)) * sizeof(float);
    if (cudaFuncSetAttribute(reverse_cross_kernel<D, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    reverse_cross_kernel<D, DV><<<dim3(b.nseg - 1, b.BH), kThreads, smem, st>>>(b, CB);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_reverse_scan(const float* src, float* dst, int BH, int H, int nseg, size_t E, const float* gamma,
                        int n, int W, int seg_chunks, int power, cudaStream_t st) {
    const size_t total = (size_t)BH * E;
    if (total == 0 || nseg <= 0) return 0;
    if (launch_pdl(reverse_scan_kernel, dim3((unsigned)((total + kThreads - 1) / kThreads)), dim3(kThreads), 0, st,
                   src, dst, BH, H, nseg, E, gamma, n, W, seg_chunks, power) != cudaSuccess)
        return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_reverse_cross(const BwdArgs& b, const float* CB, int d, int dv, cudaStream_t st) {
    if (b.nseg <= 1 || b.BH <= 0) return 0;
#define HLA2_RCROSS(DD, VV) \
    if (d == DD && dv == VV) return launch_reverse_cross_t<DD, VV>(b, CB, st);
    HLA2_RCROSS(16, 16) HLA2_RCROSS(16, 32) HLA2_RCROSS(16, 64) HLA2_RCROSS(16, 128)
    HLA2_RCROSS(32, 16) HLA2_RCROSS(32, 32) HLA2_RCROSS(32, 64) HLA2_RCROSS(32, 128)
    HLA2_RCROSS(64, 16) HLA2_RCROSS(64, 32) HLA2_RCROSS(64, 64) HLA2_RCROSS(64, 128)
    HLA2_RCROSS(128, 16) HLA2_RCROSS(128, 32) HLA2_RCROSS(128, 64) HLA2_RCROSS(128, 128)
    HLA2_RCROSS(16, 48) HLA2_RCROSS(16, 80) HLA2_RCROSS(16, 144)
    HLA2_RCROSS(32, 48) HLA2_RCROSS(32, 80) HLA2_RCROSS(32, 144)
    HLA2_RCROSS(64, 48) HLA2_RCROSS(64, 80) HLA2_RCROSS(64, 144)
    HLA2_RCROSS(128, 48) HLA2_RCROSS(128, 80) HLA2_RCROSS(128, 144)
#undef HLA2_RCROSS
    return -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(scan)
