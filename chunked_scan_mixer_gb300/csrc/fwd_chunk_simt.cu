// SIMT chunk kernel of the masked HLA-2 forward: fp32 arithmetic on shared-memory
// tiles, runtime shapes.  Same per-chunk algebra as the tensor-core kernel
// (fwd_chunk_mma.cuh), written as plain loops; it serves float32 inputs (where bf16
// tensor-core operands would not meet a 1e-4 relative error) and bf16 shapes the
// tensor-core kernel does not cover.  With a.unmasked it computes the unmasked output
// q^T S C (section summary §3, §4.1): Z and y then hold C and m, the second product is
// (P Q^T) * [j <= r] g^(r-j), and the carry term is g^(r+1) P C0.
#include "kernels.h"

namespace hla2 {

namespace {

struct SimtLayout {
    size_t Q, K, V, AB, P, S, Z, C, y, m, gp, den, total;
};

__host__ __device__ inline SimtLayout simt_layout(int D, int DV, int W, bool cm) {
    SimtLayout L;
    size_t o = 0;
    L.Q = o; o += (size_t)W * D;
    L.K = o; o += (size_t)W * D;
    L.V = o; o += (size_t)W * DV;
    L.AB = o; o += (size_t)W * W;
    L.P = o; o += (size_t)W * D;
    L.S = o; o += (size_t)D * D;
    L.Z = o; o += (size_t)D * DV;
    L.C = o; o += cm ? (size_t)D * DV : 0;
    L.y = o; o += D;
    L.m = o; o += D;
    L.gp = o; o += 2 * (size_t)W + 2;
    L.den = o; o += W;
    L.total = o;
    return L;
}

constexpr int kSimtThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kSimtThreads)
    fwd_chunk_simt_kernel(const ChunkArgs a, int D, int DV, int W, int summary, int cm) {
    extern __shared__ __align__(16) float sm[];
    const SimtLayout L = simt_layout(D, DV, W, cm != 0);
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Vs = sm + L.V, *AB = sm + L.AB, *Ps = sm + L.P;
    float *S = sm + L.S, *Z = sm + L.Z, *C = sm + L.C, *y = sm + L.y, *m = sm + L.m;
    float *gp = sm + L.gp, *den = sm + L.den;
    const int tid = threadIdx.x, NT = blockDim.x;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y, nseg = a.nseg;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const T* q = static_cast<const T*>(a.q) + (size_t)bh * a.n * D;
    const T* k = static_cast<const T*>(a.k) + (size_t)bh * a.n * D;
    const T* v = static_cast<const T*>(a.v) + (size_t)bh * a.n * DV;
    const bool um = a.unmasked != 0;
    const bool need_p = !(summary && um);  // the unmasked summary needs no p
    const int bp = um ? 1 : 2;             // decay power of the second scan

    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);

    // initial state: zero (summary) or the segment's carry-in
    const size_t sidx = (size_t)bh * nseg + seg;
    auto wsr = [&](size_t idx, int site) { return HLA2_IN(idx < a.L.total, site) ? a.ws[idx] : 0.f; };
    for (int i = tid; i < D * D; i += NT) S[i] = summary ? 0.f : wsr(a.L.Sin + sidx * D * D + i, 201);
    for (int i = tid; i < D * DV; i += NT) {
        Z[i] = summary ? 0.f : wsr(a.L.Zin + sidx * D * DV + i, 202);
        if (cm) C[i] = summary ? 0.f : wsr(a.L.Clast + (size_t)bh * D * DV + i, 203);
    }
    for (int i = tid; i < D; i += NT) {
        y[i] = summary ? 0.f : wsr(a.L.yin + sidx * D + i, 204);
        m[i] = (cm && !summary) ? wsr(a.L.mlast + (size_t)bh * D + i, 205) : 0.f;
    }

    for (int c = c_begin; c < c_end; ++c) {
        const int row0 = c * W;
        const int Wc = min(W, a.n - row0);
        __syncthreads();
        if (!summary && a.chunk_states_f32) {  // the state at this chunk start, for the backward
            const size_t cs = (size_t)(D * D + D * DV), base = ((size_t)bh * a.nchunks + c) * cs;
            float* dst = a.chunk_states_f32 + base;
            const bool ok = HLA2_IN(bh < a.BH && c < a.nchunks && base + cs <= (size_t)a.BH * a.nchunks * cs, 206);
            for (int i = tid; ok && i < D * D; i += NT) dst[i] = S[i];
            for (int i = tid; ok && i < D * DV; i += NT) dst[(size_t)D * D + i] = Z[i];
        }
        for (int i = tid; i < W * D; i += NT) {
            const int r = i / D;
            const bool in = r < Wc && HLA2_IN((size_t)row0 * D + i < (size_t)a.n * D, 207);
            Qs[i] = in ? to_f32(q[(size_t)row0 * D + i]) : 0.f;
            Ks[i] = in ? to_f32(k[(size_t)row0 * D + i]) : 0.f;
        }
        for (int i = tid; i < W * DV; i += NT)
            Vs[i] = ((i / DV) < Wc && HLA2_IN((size_t)row0 * DV + i < (size_t)a.n * DV, 208))
                        ? to_f32(v[(size_t)row0 * DV + i]) : 0.f;
        __syncthreads();

        // A~[r, i] = [i <= r] g^(r-i) q_r . k_i ; den carry term
        for (int e = tid; need_p && e < W * W; e += NT) {
            const int r = e / W, i = e % W;
            float s = 0.f;
            if (i <= r)
                for (int f = 0; f < D; ++f) s += Qs[r * D + f] * Ks[i * D + f];
            AB[e] = i <= r ? gp[r - i] * s : 0.f;
        }
        if (!summary && a.normalize && !um) {
            for (int r = tid; r < W; r += NT) {
                float s = 0.f;
                for (int f = 0; f < D; ++f) s += Qs[r * D + f] * y[f];
                den[r] = gp[2 * (r + 1)] * s;
            }
        }
        __syncthreads();

        // P = diag(g^(r+1)) Q S0 + A~ K
        for (int e = tid; need_p && e < W * D; e += NT) {
            const int r = e / D, f = e % D;
            float s0 = 0.f, s1 = 0.f;
            for (int x = 0; x < D; ++x) s0 += Qs[r * D + x] * S[x * D + f];
            for (int i = 0; i <= r; ++i) s1 += AB[r * W + i] * Ks[i * D + f];
            Ps[e] = gp[r + 1] * s0 + s1;
        }
        __syncthreads();

        if (!summary && a.out) {
            if (um && a.normalize) {  // unmasked denominator carry g^(r+1) p_r . m0
                for (int r = tid; r < W; r += NT) {
                    float s = 0.f;
                    for (int f = 0; f < D; ++f) s += Ps[r * D + f] * y[f];
                    den[r] = gp[r + 1] * s;
                }
            }
            // B~[r, j] = [j <= r] g^(2(r-j)) q_r . p_j   (unmasked: g^(r-j) p_r . q_j)
            for (int e = tid; e < W * W; e += NT) {
                const int r = e / W, j = e % W;
                float s = 0.f;
                if (j <= r) {
                    const float* x0 = um ? Ps + r * D : Qs + r * D;
                    const float* x1 = um ? Qs + j * D : Ps + j * D;
                    for (int f = 0; f < D; ++f) s += x0[f] * x1[f];
                }
                AB[e] = j <= r ? gp[bp * (r - j)] * s : 0.f;
            }
            __syncthreads();
            if (a.normalize) {
                for (int r = tid; r < W; r += NT) {
                    float s = 0.f;
                    for (int j = 0; j <= r; ++j) s += AB[r * W + j];
                    den[r] += s;
                }
                __syncthreads();
            }
            // O = diag(g^(2(r+1))) Q Z0 + B~ V   (unmasked: diag(g^(r+1)) P C0 + B~ V)
            T* out = static_cast<T*>(a.out) + ((size_t)bh * a.n + row0) * DV;
            const float* lhs = um ? Ps : Qs;
            for (int e = tid; e < Wc * DV; e += NT) {
                const int r = e / DV, x = e % DV;
                float s0 = 0.f, s1 = 0.f;
                for (int f = 0; f < D; ++f) s0 += lhs[r * D + f] * Z[f * DV + x];
                for (int j = 0; j <= r; ++j) s1 += AB[r * W + j] * Vs[j * DV + x];
                float o = gp[bp * (r + 1)] * s0 + s1;
                if (a.normalize) o /= (den[r] + a.eps);
                if (HLA2_IN(row0 + r < a.n && bh < a.BH, 209)) out[e] = from_f32<T>(o);
            }
            __syncthreads();
        }

        // state updates (each element owned by one thread); unmasked, Z and y take the
        // query-value and query-mass increments with decay g
        const float rho = gp[Wc], rho2 = gp[bp * Wc];
        const float* zl = um ? Qs : Ps;  // left factor of the Z and y increments
        for (int e = tid; e < D * D; e += NT) {
            const int x = e / D, f = e % D;
            float s = 0.f;
            for (int i = 0; i < Wc; ++i) s += gp[Wc - 1 - i] * Ks[i * D + x] * Ks[i * D + f];
            S[e] = rho * S[e] + s;
        }
        for (int e = tid; e < D * DV; e += NT) {
            const int x = e / DV, f = e % DV;
            float s = 0.f, sc = 0.f;
            for (int j = 0; j < Wc; ++j) {
                s += gp[bp * (Wc - 1 - j)] * zl[j * D + x] * Vs[j * DV + f];
                if (cm) sc += gp[Wc - 1 - j] * Qs[j * D + x] * Vs[j * DV + f];
            }
            Z[e] = rho2 * Z[e] + s;
            if (cm) C[e] = rho * C[e] + sc;
        }
        for (int x = tid; x < D; x += NT) {
            float s = 0.f, sm_ = 0.f;
            for (int j = 0; j < Wc; ++j) {
                s += gp[bp * (Wc - 1 - j)] * zl[j * D + x];
                sm_ += gp[Wc - 1 - j] * Qs[j * D + x];
            }
            y[x] = rho2 * y[x] + s;
            m[x] = rho * m[x] + sm_;
        }
    }
    __syncthreads();

    float *dS = nullptr, *dC = nullptr, *dZ = nullptr, *dm = nullptr, *dy = nullptr;
    if (summary) {
        const size_t si = (size_t)bh * a.nsum + seg;
        dS = a.ws + a.L.SB + si * D * D;
        dC = a.ws + a.L.CB + si * D * DV;
        dZ = a.ws + a.L.ZB + si * D * DV;
        dm = a.ws + a.L.mB + si * D;
        dy = a.ws + a.L.yB + si * D;
    } else if ((cm || um) && seg == nseg - 1 && a.want_final) {
        const RawOff ro = raw_off(D, DV);
        float* base = a.ws + a.L.fin + (size_t)bh * raw_state_floats(D, DV);
        dS = base + ro.S;
        dC = base + ro.C;
        dZ = base + ro.Z;
        dm = base + ro.m;
        dy = base + ro.y;
    }
    if (dS && HLA2_IN((size_t)(dy + D - a.ws) <= a.L.total && dS >= a.ws, 210)) {
        for (int i = tid; i < D * D; i += NT) dS[i] = S[i];
        for (int i = tid; i < D * DV; i += NT) {
            dZ[i] = Z[i];
            if (cm) dC[i] = C[i];
        }
        for (int i = tid; i < D; i += NT) {
            dm[i] = m[i];
            dy[i] = y[i];
        }
    }
}

}  // namespace

size_t fwd_chunk_simt_smem(int d, int dv, int W, bool track_cm) {
    return simt_layout(d, dv, W, track_cm).total * sizeof(float);
}

int launch_fwd_chunk_simt(const ChunkArgs& a, int d, int dv, int W, bool summary, bool track_cm,
                          bool is_bf16, cudaStream_t st) {
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
    const bool cm = !a.unmasked && (summary || track_cm);
    const size_t smem = fwd_chunk_simt_smem(d, dv, W, cm);
    dim3 grid(a.nseg_launch, a.BH), block(kSimtThreads);
    cudaError_t e;
    if (is_bf16) {
        auto kfn = fwd_chunk_simt_kernel<bf16>;
        e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) kfn<<<grid, block, smem, st>>>(a, d, dv, W, summary, cm);
    } else {
        auto kfn = fwd_chunk_simt_kernel<float>;
        e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) kfn<<<grid, block, smem, st>>>(a, d, dv, W, summary, cm);
    }
    if (e != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(fwd_simt)
