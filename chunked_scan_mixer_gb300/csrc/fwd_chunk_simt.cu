// SIMT chunk kernel of the masked HLA-2 forward: float32 arithmetic on shared-memory
// tiles, runtime shapes.  Same per-chunk algebra as the tensor-core kernels
// (fwd_chunk_mma.cuh); it serves float32 inputs (where bf16 tensor-core operands would not
// meet a 1e-4 relative error) and bf16 shapes the tensor-core kernels do not cover.  With
// a.unmasked it computes the unmasked output q^T S C (section summary §3, §4.1): Z and y
// then hold C and m, the second product is (P Q^T) * [j <= r] g^(r-j), and the carry term
// is g^(r+1) P C0.
//
// Per chunk of width W (rows r < Wc, state S0, Z0, y0 at the chunk start, g the decay):
//   A~[r, i] = [i <= r] g^(r-i) q_r . k_i
//   P        = diag(g^(r+1)) Q S0 + A~ K                       (p_r = S_r q_r)
//   B~[r, j] = [j <= r] g^(2(r-j)) q_r . p_j
//   O        = diag(g^(2(r+1))) Q Z0 + B~ V                    (o_r = Z_r^T q_r)
//   den_r    = g^(2(r+1)) q_r . y0 + sum_j B~[r, j]           (normalised: o_r / (den_r + eps))
//   S <- g^Wc S0 + K~^T K,  Z <- g^(2Wc) Z0 + P~^T V,  y <- g^(2Wc) y0 + sum_j g^(2(Wc-1-j)) p_j
// with K~, P~ the rows scaled by their decay to the chunk end; C and m (summaries and the
// final state) take q v^T and q with decay g.  Every product runs through the register-tiled
// helpers of simt_tile.cuh: a thread owns an RM x 4 block of the output.
#include "kernels.h"
#include "simt_tile.cuh"

namespace hla2 {

namespace {

using simt::kThreads;

// Shared-memory tiles (floats).  Q, K, V, P row-major with padded rows; T holds K^T for the
// key Gram, then P^T (masked) or Q^T (unmasked) for the second Gram; AB holds A~, then B~.
// S and Z (and C while it fits without lowering the CTAs an SM holds; else C accumulates in the
// slot it is written to) are row-major without padding: they are read only as the B operand of
// a product, or updated by the thread that owns a block.
struct SimtLayout {
    int ldD, ldV, ldW;
    bool c_smem;
    size_t Q, K, T, V, AB, P, S, Z, C, y, m, den, gp, total;
};

__host__ __device__ inline SimtLayout simt_layout(int D, int DV, int W, bool cm) {
    SimtLayout L;
    L.ldD = simt::pad(D);
    L.ldV = simt::pad(DV);
    L.ldW = simt::pad(W);
    size_t o = 0;
    L.Q = o;   o += (size_t)W * L.ldD;
    L.K = o;   o += (size_t)W * L.ldD;
    L.T = o;   o += (size_t)D * L.ldW;
    L.V = o;   o += (size_t)W * L.ldV;
    L.AB = o;  o += (size_t)W * L.ldW;
    L.P = o;   o += (size_t)W * L.ldD;
    L.S = o;   o += (size_t)D * D;
    L.Z = o;   o += (size_t)D * DV;
    L.y = o;   o += D;
    L.m = o;   o += D;
    L.den = o; o += W;
    L.gp = o;  o += 2 * (size_t)W + 2;
    o = (o + 3) & ~(size_t)3;
    L.c_smem = cm && simt::fits_beside(o, (size_t)D * DV, kSimtFwdCtas);
    L.C = o;   o += L.c_smem ? (size_t)D * DV : 0;
    L.total = o;
    return L;
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&r)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&r)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    r[0] = v.x;
    r[1] = v.y;
    r[2] = v.z;
    r[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<bf16>(const bf16* p, float (&r)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
    r[0] = __low2float(a);
    r[1] = __high2float(a);
    r[2] = __low2float(b);
    r[3] = __high2float(b);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, kSimtFwdCtas)
    fwd_chunk_simt_kernel(const ChunkArgs a, int D, int DV, int W, int summary, int cm) {
    extern __shared__ __align__(16) float sm[];
    const SimtLayout L = simt_layout(D, DV, W, cm != 0);
    const int ldD = L.ldD, ldV = L.ldV, ldW = L.ldW;
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Ts = sm + L.T, *Vs = sm + L.V, *AB = sm + L.AB, *Ps = sm + L.P;
    float *S = sm + L.S, *Z = sm + L.Z, *y = sm + L.y, *m = sm + L.m, *den = sm + L.den, *gp = sm + L.gp;
    const int tid = threadIdx.x;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y, nseg = a.nseg;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const T* q = static_cast<const T*>(a.q) + (size_t)bh * a.n * D;
    const T* k = static_cast<const T*>(a.k) + (size_t)bh * a.n * D;
    const T* v = static_cast<const T*>(a.v) + (size_t)bh * a.n * DV;
    const bool um = a.unmasked != 0;
    const bool need_p = !(summary && um);          // the unmasked summary needs no p
    const bool out_pass = !summary && a.out != nullptr;
    const bool norm = out_pass && a.normalize;
    const int bp = um ? 1 : 2;                     // decay power of the second scan
    // The final raw state is written by the last segment of an output pass that wants it.
    const bool final_seg = !summary && (cm || um) && seg == nseg - 1 && a.want_final;
    // C (masked only) is kept where it is written: summaries and the final state.
    const bool keep_c = cm && (summary || final_seg);

    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += kThreads) gp[i] = pow_decay(log2g, (float)i);

    // destination of the summaries or of the final state (also where a large C accumulates)
    float *dS = nullptr, *dC = nullptr, *dZ = nullptr, *dm = nullptr, *dy = nullptr;
    if (summary) {
        const size_t si = (size_t)bh * a.nsum + seg;
        dS = a.ws + a.L.SB + si * D * D;
        dC = a.ws + a.L.CB + si * D * DV;
        dZ = a.ws + a.L.ZB + si * D * DV;
        dm = a.ws + a.L.mB + si * D;
        dy = a.ws + a.L.yB + si * D;
    } else if (final_seg) {
        const RawOff ro = raw_off(D, DV);
        float* base = a.ws + a.L.fin + (size_t)bh * raw_state_floats(D, DV);
        dS = base + ro.S;
        dC = base + ro.C;
        dZ = base + ro.Z;
        dm = base + ro.m;
        dy = base + ro.y;
    }
    const bool dst_ok = dS && HLA2_IN((size_t)(dy + D - a.ws) <= a.L.total && dS >= a.ws, 210);
    float* C = L.c_smem ? sm + L.C : dC;  // row-major [D][DV]
    const bool track_c = keep_c && (L.c_smem || dst_ok);

    // initial state: zero (summary) or the segment's carry-in
    const size_t sidx = (size_t)bh * nseg + seg;
    auto wsr = [&](size_t idx, int site) { return HLA2_IN(idx < a.L.total, site) ? a.ws[idx] : 0.f; };
    for (int i = tid; i < D * D; i += kThreads) S[i] = summary ? 0.f : wsr(a.L.Sin + sidx * D * D + i, 201);
    for (int i = tid; i < D * DV; i += kThreads) {
        Z[i] = summary ? 0.f : wsr(a.L.Zin + sidx * D * DV + i, 202);
        if (track_c) C[i] = summary ? 0.f : wsr(a.L.Clast + (size_t)bh * D * DV + i, 203);
    }
    for (int i = tid; i < D; i += kThreads) {
        y[i] = summary ? 0.f : wsr(a.L.yin + sidx * D + i, 204);
        m[i] = (!summary && keep_c) ? wsr(a.L.mlast + (size_t)bh * D + i, 205) : 0.f;
    }

    for (int c = c_begin; c < c_end; ++c) {
        const int row0 = c * W;
        const int Wc = min(W, a.n - row0);
        __syncthreads();  // the previous chunk's state updates are done
        if (!summary && a.chunk_states_f32) {  // the state at this chunk start, for the backward
            const size_t cs = (size_t)(D * D + D * DV), base = ((size_t)bh * a.nchunks + c) * cs;
            float* dst = a.chunk_states_f32 + base;
            if (HLA2_IN(bh < a.BH && c < a.nchunks && base + cs <= (size_t)a.BH * a.nchunks * cs, 206)) {
                for (int i = tid; i < (D * D) / 4; i += kThreads)
                    reinterpret_cast<float4*>(dst)[i] = reinterpret_cast<const float4*>(S)[i];
                for (int i = tid; i < (D * DV) / 4; i += kThreads)
                    reinterpret_cast<float4*>(dst + (size_t)D * D)[i] = reinterpret_cast<const float4*>(Z)[i];
            }
        }
        // tiles of this chunk (rows past the end are zero); K^T beside K for the key Gram
        for (int i = tid; i < W * D; i += kThreads) {
            const int r = i / D, f = i - r * D;
            const bool in = r < Wc && HLA2_IN((size_t)row0 * D + i < (size_t)a.n * D, 207);
            const float qx = in ? to_f32(q[(size_t)row0 * D + i]) : 0.f;
            const float kx = in ? to_f32(k[(size_t)row0 * D + i]) : 0.f;
            Qs[r * ldD + f] = qx;
            Ks[r * ldD + f] = kx;
            if (need_p) Ts[f * ldW + r] = kx;
        }
        for (int i = tid; i < (W * DV) / 4; i += kThreads) {
            const int r = (4 * i) / DV, x = 4 * i - r * DV;
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            if (r < Wc && HLA2_IN((size_t)row0 * DV + 4 * i + 4 <= (size_t)a.n * DV, 208))
                load4<T>(v + (size_t)row0 * DV + 4 * i, t);
            simt::st4(Vs + r * ldV + x, t);
        }
        __syncthreads();

        // A~ = (Q K^T) * [i <= r] g^(r-i); masked denominator carry g^(2(r+1)) q_r . y0
        if (need_p) {
            simt::with_rm(W, W, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, W, [&](int m0, int n0) {
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    if (n0 < m0 + RM) simt::mac_r<RM>(acc, Qs + m0 * ldD, ldD, Ts + n0, ldW, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) {
                        const int r = m0 + i;
#pragma unroll
                        for (int b = 0; b < 4; ++b) acc[i][b] = n0 + b <= r ? gp[r - n0 - b] * acc[i][b] : 0.f;
                        simt::st4(AB + r * ldW + n0, acc[i]);
                    }
                });
            });
        }
        if (norm && !um) {
            for (int r = tid; r < W; r += kThreads) {
                float s = 0.f;
                for (int f = 0; f < D; ++f) s = fmaf(Qs[r * ldD + f], y[f], s);
                den[r] = gp[2 * (r + 1)] * s;
            }
        }
        __syncthreads();

        // P = diag(g^(r+1)) Q S0 + A~ K; P^T (masked output pass) or Q^T (unmasked) into T
        if (need_p) {
            simt::with_rm(W, D, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, D, [&](int m0, int n0) {
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, Qs + m0 * ldD, ldD, S + n0, D, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::scale_row(acc, i, gp[m0 + i + 1]);
                    simt::mac_r<RM>(acc, AB + m0 * ldW, ldW, Ks + n0, ldD, min(W, m0 + RM));
#pragma unroll
                    for (int i = 0; i < RM; ++i) {
                        simt::st4(Ps + (m0 + i) * ldD + n0, acc[i]);
                        if (out_pass && !um) {
#pragma unroll
                            for (int b = 0; b < 4; ++b) Ts[(n0 + b) * ldW + m0 + i] = acc[i][b];
                        }
                    }
                });
            });
        }
        if (out_pass && um)
            for (int i = tid; i < W * D; i += kThreads) {
                const int r = i / D, f = i - r * D;
                Ts[f * ldW + r] = Qs[r * ldD + f];
            }
        __syncthreads();

        if (out_pass) {
            if (norm && um) {  // unmasked denominator carry g^(r+1) p_r . m0
                for (int r = tid; r < W; r += kThreads) {
                    float s = 0.f;
                    for (int f = 0; f < D; ++f) s = fmaf(Ps[r * ldD + f], y[f], s);
                    den[r] = gp[r + 1] * s;
                }
            }
            // B~[r, j] = [j <= r] g^(2(r-j)) q_r . p_j   (unmasked: g^(r-j) p_r . q_j)
            const float* X0 = um ? Ps : Qs;
            simt::with_rm(W, W, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, W, [&](int m0, int n0) {
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    if (n0 < m0 + RM) simt::mac_r<RM>(acc, X0 + m0 * ldD, ldD, Ts + n0, ldW, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) {
                        const int r = m0 + i;
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            acc[i][b] = n0 + b <= r ? gp[bp * (r - n0 - b)] * acc[i][b] : 0.f;
                        simt::st4(AB + r * ldW + n0, acc[i]);
                    }
                });
            });
            __syncthreads();

            // O = diag(g^(2(r+1))) Q Z0 + B~ V   (unmasked: diag(g^(r+1)) P C0 + B~ V)
            T* out = static_cast<T*>(a.out) + ((size_t)bh * a.n + row0) * DV;
            simt::with_rm(W, DV, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, DV, [&](int m0, int n0) {
                    if (m0 >= Wc) return;
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, X0 + m0 * ldD, ldD, Z + n0, DV, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::scale_row(acc, i, gp[bp * (m0 + i + 1)]);
                    simt::mac_r<RM>(acc, AB + m0 * ldW, ldW, Vs + n0, ldV, min(W, m0 + RM));
#pragma unroll
                    for (int i = 0; i < RM; ++i) {
                        const int r = m0 + i;
                        if (r >= Wc) break;
                        if (norm) {
                            float dn = den[r];
                            for (int j = 0; j <= r; ++j) dn += AB[r * ldW + j];
                            const float dd = dn + a.eps;
#pragma unroll
                            for (int b = 0; b < 4; ++b) acc[i][b] /= dd;
                        }
                        if (HLA2_IN(row0 + r < a.n && bh < a.BH, 209)) simt::store4(out + (size_t)r * DV + n0, acc[i]);
                    }
                });
            });
            __syncthreads();  // S0 and Z0 are read above
        }

        // the state to the chunk end (the output pass skips it after its last chunk unless the
        // final state is written); each block owned by one thread
        if (!summary && c + 1 == c_end && !final_seg) continue;
        const float rho = gp[Wc], rho2 = gp[bp * Wc];
        simt::with_rm(D, D, [&](auto t) {  // S <- g^Wc S0 + K~^T K
            constexpr int RM = decltype(t)::value;
            simt::for_blocks<RM>(D, D, [&](int m0, int n0) {
                simt::Acc<RM> acc;
                simt::zero(acc);
                simt::mac_c<RM>(acc, Ks + m0, ldD, Ks + n0, ldD, 0, Wc, [&](int i) { return gp[Wc - 1 - i]; });
#pragma unroll
                for (int i = 0; i < RM; ++i) simt::decay_add4(S + (m0 + i) * D + n0, rho, acc[i]);
            });
        });
        // Z (masked: P~^T V with g^2; unmasked: Q~^T V with g) and C = Q~^T V with g
        const float* ZL = um ? Qs : Ps;
        simt::with_rm(D, DV, [&](auto t) {
            constexpr int RM = decltype(t)::value;
            simt::for_blocks<RM>(D, DV, [&](int m0, int n0) {
                simt::Acc<RM> az;
                simt::zero(az);
                if (track_c) {
                    simt::Acc<RM> ac;
                    simt::zero(ac);
#pragma unroll 2
                    for (int j = 0; j < Wc; ++j) {
                        const float4 b = simt::ldb4(Vs + n0, ldV, j);
                        float xz[RM], xc[RM];
                        simt::ldv<RM>(xz, ZL + j * ldD + m0);
                        simt::ldv<RM>(xc, Qs + j * ldD + m0);
                        simt::fma_row<RM>(az, xz, simt::scale4(b, gp[bp * (Wc - 1 - j)]));
                        simt::fma_row<RM>(ac, xc, simt::scale4(b, gp[Wc - 1 - j]));
                    }
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::decay_add4(C + (m0 + i) * DV + n0, rho, ac[i]);
                } else {
                    simt::mac_c<RM>(az, ZL + m0, ldD, Vs + n0, ldV, 0, Wc,
                                    [&](int j) { return gp[bp * (Wc - 1 - j)]; });
                }
#pragma unroll
                for (int i = 0; i < RM; ++i) simt::decay_add4(Z + (m0 + i) * DV + n0, rho2, az[i]);
            });
        });
        for (int x = tid; x < D; x += kThreads) {
            float s = 0.f, sq = 0.f;
            for (int j = 0; j < Wc; ++j) {
                s = fmaf(gp[bp * (Wc - 1 - j)], ZL[j * ldD + x], s);
                sq = fmaf(gp[Wc - 1 - j], Qs[j * ldD + x], sq);
            }
            y[x] = rho2 * y[x] + s;
            if (keep_c || um) m[x] = rho * m[x] + sq;
        }
    }
    __syncthreads();

    if (dst_ok) {
        for (int i = tid; i < D * D; i += kThreads) dS[i] = S[i];
        for (int i = tid; i < D * DV; i += kThreads) {
            dZ[i] = Z[i];
            if (cm && L.c_smem) dC[i] = C[i];
        }
        for (int i = tid; i < D; i += kThreads) {
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
    if ((d & 15) || (dv & 15) || (W & 15)) return -1;
    const bool cm = !a.unmasked && (summary || track_cm);
    const size_t smem = fwd_chunk_simt_smem(d, dv, W, cm);
    dim3 grid(a.nseg_launch, a.BH), block(kThreads);
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
