// Reverse-mode chunk scan of the AHLA forward (SIMT, float32 arithmetic; float32 or bf16
// tensors, d == dv).  Gradients of the unnormalised output, equal to those of the serial
// recurrence (page "Higher-order Linear Attention", section summary §4.2: a reverse-mode scan
// reproduces the serial recurrence's gradients; technical summary item 2 for the operator).
//
// Forward per chunk (rows r < Wc, state P0, E0 at the chunk start, decays g^i):
//   A~[r,j] = [j <= r] g^(r-j) q_r.k_j,   I[r] = g^(r+1) P0^T q_r + sum_j A~[r,j] v_j,
//   o_r = g^(r+1) E0^T q_r + sum_j A~[r,j] I_j,
//   P <- g^Wc P0 + sum_j g^(Wc-1-j) k_j v_j^T,   E <- g^Wc E0 + sum_j g^(Wc-1-j) k_j I_j^T,
//   and the segment summary R = sum_j k_j q_j^T (undecayed).
// Reverse per chunk, with Eh, Ph the adjoints of E, P at the chunk end:
//   dI[j]  = sum_{r >= j} A~[r,j] dO_r + g^(Wc-1-j) Eh^T k_j
//   dA[r,j] = [j <= r] g^(r-j) (dO_r . I_j + dI_r . v_j)
//   dq_r = g^(r+1) (E0 dO_r + P0 dI_r) + sum_j dA[r,j] k_j
//   dk_j = g^(Wc-1-j) (Eh I_j + Ph v_j) + sum_{r >= j} dA[r,j] q_r
//   dv_j = sum_{r >= j} A~[r,j] dI_r + g^(Wc-1-j) Ph^T k_j
//   Eh <- g^Wc Eh + sum_r g^(r+1) q_r dO_r^T,   Ph <- g^Wc Ph + sum_r g^(r+1) q_r dI_r^T.
// Across segments (s the later one, rho_s = g^(length of s)):
//   forward  E_in(s+1) = rho E_in(s) + E_B(s) + rho R_B(s) P_in(s)   (P: plain prefix)
//   reverse  Ph_end(s-1) = rho Ph_end(s) + Ph_B(s) + rho R_B(s)^T Eh_end(s)   (Eh: plain suffix)
// The passes: forward summaries of every segment (P_B, E_B, R_B), the forward scan, a walk
// that stores the forward state at every chunk start, reverse summaries (Eh_B, Ph_B), the
// reverse scan, and the gradient pass.  Running states live in the workspace slot of their
// segment and are updated in place, one element per thread.
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kAbThreads = 256;

struct AbSmem {
    size_t Q, K, V, O, A, I, dI, dA, gp, total;
};

__host__ __device__ inline AbSmem ab_smem(int D, int W) {
    AbSmem L;
    size_t o = 0;
    L.Q = o;  o += (size_t)W * D;
    L.K = o;  o += (size_t)W * D;
    L.V = o;  o += (size_t)W * D;
    L.O = o;  o += (size_t)W * D;
    L.A = o;  o += (size_t)W * W;
    L.I = o;  o += (size_t)W * D;
    L.dI = o; o += (size_t)W * D;
    L.dA = o; o += (size_t)W * W;
    L.gp = o; o += 2 * (size_t)W + 2;
    L.total = o;
    return L;
}

enum AbMode { kFwdSummary = 0, kFwdStates = 1, kRevSummary = 2, kGrad = 3 };

template <typename T, int MODE>
__global__ void __launch_bounds__(kAbThreads) ahla_bwd_kernel(const AhlaBwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int D = a.d, W = a.W;
    const AbSmem L = ab_smem(D, W);
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Vs = sm + L.V, *Os = sm + L.O, *As = sm + L.A;
    float *Is = sm + L.I, *dIs = sm + L.dI, *dAs = sm + L.dA, *gp = sm + L.gp;
    const int tid = threadIdx.x, NT = blockDim.x;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const size_t hq = (size_t)bh * a.n, dd = (size_t)D * D, sidx = (size_t)bh * a.nseg + seg;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);
    const T* q = static_cast<const T*>(a.q) + hq * D;
    const T* k = static_cast<const T*>(a.k) + hq * D;
    const T* v = static_cast<const T*>(a.v) + hq * D;
    const T* dO = static_cast<const T*>(a.dout) + hq * D;
    constexpr bool FWD = MODE == kFwdSummary || MODE == kFwdStates;
    constexpr bool NEED_I = MODE != kRevSummary;
    constexpr bool NEED_DO = MODE == kRevSummary || MODE == kGrad;

    // running states of this segment
    float *P = nullptr, *E = nullptr, *R = nullptr, *Eh = nullptr, *Ph = nullptr;
    if (MODE == kFwdSummary) {
        P = a.ws + a.PB + sidx * dd;
        E = a.ws + a.EB + sidx * dd;
        R = a.ws + a.RB + sidx * dd;
        for (int i = tid; i < D * D; i += NT) P[i] = E[i] = R[i] = 0.f;
    } else if (MODE == kRevSummary || MODE == kGrad) {
        Eh = a.ws + (MODE == kRevSummary ? a.EhB : a.Eh_end) + sidx * dd;
        Ph = a.ws + (MODE == kRevSummary ? a.PhB : a.Ph_end) + sidx * dd;
        if (MODE == kRevSummary)
            for (int i = tid; i < D * D; i += NT) Eh[i] = Ph[i] = 0.f;
    } else if (c_begin < c_end) {  // kFwdStates: the carry is the state at the segment's first chunk
        float* st = a.ws + a.states + ((size_t)bh * a.nchunks + c_begin) * 2 * dd;
        for (int i = tid; i < D * D; i += NT) {
            st[i] = a.ws[a.Pin + sidx * dd + i];
            st[dd + i] = a.ws[a.Ein + sidx * dd + i];
        }
    }

    for (int it = 0; it < c_end - c_begin; ++it) {
        const int c = FWD ? c_begin + it : c_end - 1 - it;
        const int row0 = c * W, Wc = min(W, a.n - row0);
        if (MODE == kFwdStates || MODE == kGrad) {
            P = a.ws + a.states + ((size_t)bh * a.nchunks + c) * 2 * dd;  // state at this chunk start
            E = P + dd;
        }
        __syncthreads();  // the previous chunk's readers of the tiles and states are done
        for (int i = tid; i < W * D; i += NT) {
            const bool ok = i / D < Wc;
            Qs[i] = ok ? to_f32(q[(size_t)row0 * D + i]) : 0.f;
            Ks[i] = ok ? to_f32(k[(size_t)row0 * D + i]) : 0.f;
            Vs[i] = ok ? to_f32(v[(size_t)row0 * D + i]) : 0.f;
            if (NEED_DO) Os[i] = ok ? to_f32(dO[(size_t)row0 * D + i]) : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < W * W; e += NT) {  // A~
            const int r = e / W, j = e % W;
            float s = 0.f;
            if (j <= r)
                for (int f = 0; f < D; ++f) s += Qs[r * D + f] * Ks[j * D + f];
            As[e] = j <= r ? gp[r - j] * s : 0.f;
        }
        __syncthreads();
        if (NEED_I) {  // I = g^(r+1) P0^T q_r + A~ V
            for (int e = tid; e < W * D; e += NT) {
                const int r = e / D, x = e % D;
                float s0 = 0.f, s1 = 0.f;
                for (int f = 0; f < D; ++f) s0 += Qs[r * D + f] * P[(size_t)f * D + x];
                for (int j = 0; j <= r; ++j) s1 += As[r * W + j] * Vs[j * D + x];
                Is[e] = r < Wc ? gp[r + 1] * s0 + s1 : 0.f;
            }
            __syncthreads();
        }
        if (NEED_DO) {  // dI (uses the end-of-chunk Eh)
            for (int e = tid; e < W * D; e += NT) {
                const int j = e / D, x = e % D;
                float s0 = 0.f, s1 = 0.f;
                for (int r = j; r < Wc; ++r) s1 += As[r * W + j] * Os[r * D + x];
                if (j < Wc)
                    for (int f = 0; f < D; ++f) s0 += Eh[(size_t)f * D + x] * Ks[j * D + f];
                dIs[e] = j < Wc ? gp[Wc - 1 - j] * s0 + s1 : 0.f;
            }
            __syncthreads();
        }
        if (MODE == kGrad) {
            for (int e = tid; e < W * W; e += NT) {  // dA (decay and mask folded in)
                const int r = e / W, j = e % W;
                float s = 0.f;
                if (j <= r)
                    for (int x = 0; x < D; ++x) s += Os[r * D + x] * Is[j * D + x] + dIs[r * D + x] * Vs[j * D + x];
                dAs[e] = j <= r ? gp[r - j] * s : 0.f;
            }
            __syncthreads();
            T* gq = static_cast<T*>(a.dq) + (hq + row0) * D;
            T* gk = static_cast<T*>(a.dk) + (hq + row0) * D;
            T* gv = static_cast<T*>(a.dv) + (hq + row0) * D;
            for (int e = tid; e < Wc * D; e += NT) {
                const int r = e / D, f = e % D;
                float s0 = 0.f, s1 = 0.f;
                for (int x = 0; x < D; ++x)
                    s0 += E[(size_t)f * D + x] * Os[r * D + x] + P[(size_t)f * D + x] * dIs[r * D + x];
                for (int j = 0; j <= r; ++j) s1 += dAs[r * W + j] * Ks[j * D + f];
                gq[e] = from_f32<T>(gp[r + 1] * s0 + s1);
            }
            for (int e = tid; e < Wc * D; e += NT) {
                const int j = e / D, f = e % D;
                float s0 = 0.f, s1 = 0.f;
                for (int x = 0; x < D; ++x)
                    s0 += Eh[(size_t)f * D + x] * Is[j * D + x] + Ph[(size_t)f * D + x] * Vs[j * D + x];
                for (int r = j; r < Wc; ++r) s1 += dAs[r * W + j] * Qs[r * D + f];
                gk[e] = from_f32<T>(gp[Wc - 1 - j] * s0 + s1);
            }
            for (int e = tid; e < Wc * D; e += NT) {
                const int j = e / D, x = e % D;
                float s0 = 0.f, s1 = 0.f;
                for (int f = 0; f < D; ++f) s0 += Ph[(size_t)f * D + x] * Ks[j * D + f];
                for (int r = j; r < Wc; ++r) s1 += As[r * W + j] * dIs[r * D + x];
                gv[e] = from_f32<T>(gp[Wc - 1 - j] * s0 + s1);
            }
            __syncthreads();  // every read of the carries is done before they move
        }

        // ---- state updates, one element per thread ----------------------------------------
        const float rho = gp[Wc];
        if (MODE == kFwdSummary || (MODE == kFwdStates && c + 1 < c_end)) {
            float* Pn = MODE == kFwdSummary ? P : P + 2 * dd;  // kFwdStates: the next chunk's slot
            float* En = MODE == kFwdSummary ? E : E + 2 * dd;
            for (int e = tid; e < D * D; e += NT) {
                const int f = e / D, x = e % D;
                float sp = 0.f, se = 0.f;
                for (int j = 0; j < Wc; ++j) {
                    const float w = gp[Wc - 1 - j] * Ks[j * D + f];
                    sp += w * Vs[j * D + x];
                    se += w * Is[j * D + x];
                }
                Pn[e] = rho * P[e] + sp;
                En[e] = rho * E[e] + se;
                if (MODE == kFwdSummary) {
                    float sr = 0.f;
                    for (int j = 0; j < Wc; ++j) sr += Ks[j * D + f] * Qs[j * D + x];
                    R[e] += sr;
                }
            }
        } else if (MODE == kRevSummary || MODE == kGrad) {
            for (int e = tid; e < D * D; e += NT) {
                const int f = e / D, x = e % D;
                float se = 0.f, sp = 0.f;
                for (int r = 0; r < Wc; ++r) {
                    const float w = gp[r + 1] * Qs[r * D + f];
                    se += w * Os[r * D + x];
                    sp += w * dIs[r * D + x];
                }
                Eh[e] = rho * Eh[e] + se;
                Ph[e] = rho * Ph[e] + sp;
            }
        }
    }
}

// dst[s] += rho_s op(R_B[s]) Y[s] for s in [s0, s0 + grid.x), op = R (forward, Y = P_in) or
// R^T (reverse, Y = Eh_end); rho_s = g^(length of segment s).
__global__ void __launch_bounds__(kAbThreads)
    ahla_seg_cross_kernel(const AhlaBwdArgs a, size_t dst_off, size_t y_off, int s0, int transpose) {
    const int s = s0 + blockIdx.x, bh = blockIdx.y, D = a.d;
    const size_t dd = (size_t)D * D, si = (size_t)bh * a.nseg + s;
    const float* R = a.ws + a.RB + si * dd;
    const float* Y = a.ws + y_off + si * dd;
    float* dst = a.ws + dst_off + si * dd;
    const long start = (long)s * a.seg_chunks * a.W, len = (long)a.seg_chunks * a.W;
    const int L = (int)(a.n - start < len ? a.n - start : len);
    const float rho = pow_decay(log2f(head_decay(a.gamma, bh, a.H)), (float)L);
    for (int e = threadIdx.x; e < D * D; e += kAbThreads) {
        const int f = e / D, x = e % D;
        float acc = 0.f;
        for (int j = 0; j < D; ++j) acc += (transpose ? R[(size_t)j * D + f] : R[(size_t)f * D + j]) * Y[(size_t)j * D + x];
        dst[e] += rho * acc;
    }
}

__global__ void __launch_bounds__(kAbThreads) ahla_bwd_init_kernel(const AhlaBwdArgs a) {
    const size_t dd = (size_t)a.d * a.d, s0 = (size_t)blockIdx.x * a.nseg;
    if (blockIdx.x == 0 && threadIdx.x == 0) *reinterpret_cast<int*>(a.ws) = 0;
    for (size_t i = threadIdx.x; i < dd; i += kAbThreads) a.ws[a.Pin + s0 * dd + i] = a.ws[a.Ein + s0 * dd + i] = 0.f;
}

template <typename T, int MODE>
int ab_pass(const AhlaBwdArgs& a, cudaStream_t st) {
    const size_t smem = ab_smem(a.d, a.W).total * sizeof(float);
    auto kfn = ahla_bwd_kernel<T, MODE>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
    kfn<<<dim3(a.nseg, a.BH), kAbThreads, smem, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename T>
int ahla_backward_t(const AhlaBwdArgs& a, cudaStream_t st) {
    const size_t dd = (size_t)a.d * a.d, hs = (size_t)a.nseg * dd;
    const int steps = a.nseg - 1, seg_tokens = a.seg_chunks * a.W;
    auto ok = [] { return cudaPeekAtLastError() == cudaSuccess; };
    ahla_bwd_init_kernel<<<a.BH, kAbThreads, 0, st>>>(a);
    if (!ok() || ab_pass<T, kFwdSummary>(a, st)) return -1;
    if (steps > 0) {
        if (launch_linear_scan(a.ws + a.PB, a.ws + a.Pin, a.BH, a.H, steps, dd, hs, hs, true, a.gamma, seg_tokens, 1,
                               st))
            return -1;
        ahla_seg_cross_kernel<<<dim3(steps, a.BH), kAbThreads, 0, st>>>(a, a.EB, a.Pin, 0, 0);
        if (!ok() || launch_linear_scan(a.ws + a.EB, a.ws + a.Ein, a.BH, a.H, steps, dd, hs, hs, true, a.gamma,
                                        seg_tokens, 1, st))
            return -1;
    }
    if (ab_pass<T, kFwdStates>(a, st) || ab_pass<T, kRevSummary>(a, st)) return -1;
    if (launch_reverse_scan(a.ws + a.EhB, a.ws + a.Eh_end, a.BH, a.H, a.nseg, dd, a.gamma, a.n, a.W, a.seg_chunks, 1,
                            st))
        return -1;
    if (steps > 0) {
        ahla_seg_cross_kernel<<<dim3(steps, a.BH), kAbThreads, 0, st>>>(a, a.PhB, a.Eh_end, 1, 1);
        if (!ok()) return -1;
    }
    if (launch_reverse_scan(a.ws + a.PhB, a.ws + a.Ph_end, a.BH, a.H, a.nseg, dd, a.gamma, a.n, a.W, a.seg_chunks, 1,
                            st))
        return -1;
    return ab_pass<T, kGrad>(a, st);
}

}  // namespace

size_t ahla_bwd_smem(int d, int W) { return ab_smem(d, W).total * sizeof(float); }

AhlaBwdLayout ahla_bwd_layout(int BH, int nseg, int nchunks, int d) {
    AhlaBwdLayout L;
    const size_t per = (size_t)BH * nseg * d * d;
    size_t o = kStatusFloats;
    L.PB = o;     o = align64(o + per);
    L.EB = o;     o = align64(o + per);
    L.RB = o;     o = align64(o + per);
    L.Pin = o;    o = align64(o + per);
    L.Ein = o;    o = align64(o + per);
    L.EhB = o;    o = align64(o + per);
    L.PhB = o;    o = align64(o + per);
    L.Eh_end = o; o = align64(o + per);
    L.Ph_end = o; o = align64(o + per);
    L.states = o; o = align64(o + (size_t)BH * nchunks * 2 * d * d);
    L.total = o;
    return L;
}

int launch_ahla_backward(const AhlaBwdArgs& a, bool is_bf16, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    return is_bf16 ? ahla_backward_t<bf16>(a, st) : ahla_backward_t<float>(a, st);
}

}  // namespace hla2
