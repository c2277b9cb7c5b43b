// float32 reverse-mode chunk kernel of the masked HLA-2 backward (SIMT): the same per-chunk
// algebra as the bf16 tensor-core kernel (bwd_chunk_mma.cuh), in float32 for float32 inputs
// of any d, dv in {16, 32, 64, 128}.  Gradients of the unnormalised output, equal to those of
// the serial recurrence (page "Higher-order Linear Attention", section summary §4.2: a
// reverse-mode scan reproduces the serial recurrence's gradients).  With p_t = S_t q_t,
// Z_t = g^2 Z_{t-1} + p_t v_t^T, o_t = q_t^T Z_t the adjoint is
//     Zh_t = q_t dO_t^T + g^2 Zh_{t+1},   dp_t = Zh_t v_t,   Sh_t = dp_t q_t^T + g Sh_{t+1}
//     dq_t = Z_t dO_t + S_t dp_t,   dv_t = Zh_t^T p_t,   dk_t = (Sh_t + Sh_t^T) k_t
// and per chunk (rows r < Wc, forward state S0, Z0 at the chunk start, reverse carries Zh,
// Sh at the chunk end):
//   A~[r,i] = [i <= r] g^(r-i) q_r.k_i           D~[r,j] = [j <= r] g^(2(r-j)) dO_r.v_j
//   P[r]    = g^(r+1) S0^T q_r + sum_i A~[r,i] k_i
//   dP[j]   = g^(2(Wc-1-j)) Zh v_j + sum_{r >= j} D~[r,j] q_r
//   B~[r,j] = [j <= r] g^(2(r-j)) q_r.p_j         dA~[r,i] = [i <= r] g^(r-i) dP_r.k_i
//   dV[j]   = g^(2(Wc-1-j)) Zh^T p_j + sum_{r >= j} B~[r,j] dO_r
//   dQ[r]   = g^(r+1) (g^(r+1) Z0 dO_r + S0^T dP_r) + sum_j D~[r,j] p_j + sum_i dA~[r,i] k_i
//   dK[i]   = g^(Wc-1-i) (Sh + Sh^T) k_i + sum_{r >= i} (A~[r,i] dP_r + dA~[r,i] q_r)
//   Zh <- g^(2Wc) Zh + sum_r g^(2(r+1)) q_r dO_r^T,   Sh <- g^Wc Sh + sum_j g^(j+1) dP_j q_j^T
// One CTA walks one segment's chunks from the last to the first.  RSUM mode starts from zero
// carries, keeps only what the reverse scan needs (D~, dP and the carry updates) and stores
// the segment's (Zh, Sh).  The gradient pass starts from the carries at the segment end and
// only ever needs Sh + Sh^T, so it carries that symmetric sum (its update is the symmetric
// part of the one above, doubled).  The forward states S0, Z0 come from the float32
// state-export pass of the forward kernel.  Every product runs through the register-tiled
// helpers of simt_tile.cuh.
#include "kernels.h"
#include "simt_tile.cuh"

namespace hla2 {

namespace {

using simt::kThreads;

// Shared-memory tiles (floats): the chunk's Q, K, V, dO, P, dP row-major with padded rows;
// K^T, V^T, P^T, dP^T; the four W x W matrices; Z0^T; and, while they fit without lowering
// the CTAs an SM holds, S0 (else read from the exported states) and the carries Zh (row-major [D][DV], padded rows: it is also read as an
// A operand) and Sh (the symmetric sum in the gradient pass), else those stay in their
// workspace slots.
struct BsLayout {
    int ldD, ldV, ldW;
    bool st_smem;
    bool s0_smem;
    size_t Q, K, V, O, P, dP, Kt, Vt, Pt, dPt, At, Dt, Bt, dAt, Z0t, S0, Zh, Sh, gp, total;
};

__host__ __device__ inline BsLayout bs_layout(int D, int DV, int W) {
    BsLayout L;
    L.ldD = simt::pad(D);
    L.ldV = simt::pad(DV);
    L.ldW = simt::pad(W);
    size_t o = 0;
    L.Q = o;   o += (size_t)W * L.ldD;
    L.K = o;   o += (size_t)W * L.ldD;
    L.V = o;   o += (size_t)W * L.ldV;
    L.O = o;   o += (size_t)W * L.ldV;
    L.P = o;   o += (size_t)W * L.ldD;
    L.dP = o;  o += (size_t)W * L.ldD;
    L.Kt = o;  o += (size_t)D * L.ldW;
    L.Vt = o;  o += (size_t)DV * L.ldW;
    L.Pt = o;  o += (size_t)D * L.ldW;
    L.dPt = o; o += (size_t)D * L.ldW;
    L.At = o;  o += (size_t)W * L.ldW;
    L.Dt = o;  o += (size_t)W * L.ldW;
    L.Bt = o;  o += (size_t)W * L.ldW;
    L.dAt = o; o += (size_t)W * L.ldW;
    L.Z0t = o; o += (size_t)DV * L.ldD;
    L.gp = o;  o += 2 * (size_t)W + 2;
    o = (o + 3) & ~(size_t)3;
    L.s0_smem = simt::fits_beside(o, (size_t)D * D, kSimtBwdCtas);
    L.S0 = o;  o += L.s0_smem ? (size_t)D * D : 0;
    L.st_smem = simt::fits_beside(o, (size_t)D * L.ldV + (size_t)D * D, kSimtBwdCtas);
    L.Zh = o;  o += L.st_smem ? (size_t)D * L.ldV : 0;
    L.Sh = o;  o += L.st_smem ? (size_t)D * D : 0;
    L.total = o;
    return L;
}

// M x M lower-triangular product into T: T[r][c] = [c <= r] gp[pw (r - c)] sum_k A(r, k) B(k, c)
// with A row-major (lda) and B row-major over c (ldb).
__device__ __forceinline__ void tri_gram(float* T, int ldt, const float* A, int lda, const float* B, int ldb, int M,
                                         int K, const float* gp, int pw) {
    simt::with_rm(M, M, [&](auto t) {
        constexpr int RM = decltype(t)::value;
        simt::for_blocks<RM>(M, M, [&](int m0, int n0) {
            simt::Acc<RM> acc;
            simt::zero(acc);
            if (n0 < m0 + RM) simt::mac_r<RM>(acc, A + m0 * lda, lda, B + n0, ldb, K);
#pragma unroll
            for (int i = 0; i < RM; ++i) {
                const int r = m0 + i;
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[i][b] = n0 + b <= r ? gp[pw * (r - n0 - b)] * acc[i][b] : 0.f;
                simt::st4(T + r * ldt + n0, acc[i]);
            }
        });
    });
}

template <bool RSUM>
__global__ void __launch_bounds__(kThreads, kSimtBwdCtas) bwd_chunk_simt_kernel(const BwdArgsF a, int D, int DV) {
    extern __shared__ __align__(16) float sm[];
    const int W = a.W;
    const BsLayout L = bs_layout(D, DV, W);
    const int ldD = L.ldD, ldV = L.ldV, ldW = L.ldW;
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Vs = sm + L.V, *Os = sm + L.O, *Ps = sm + L.P, *dPs = sm + L.dP;
    float *Kt = sm + L.Kt, *Vt = sm + L.Vt, *Pt = sm + L.Pt, *dPt = sm + L.dPt;
    float *At = sm + L.At, *Dt = sm + L.Dt, *Bt = sm + L.Bt, *dAt = sm + L.dAt, *Z0t = sm + L.Z0t, *gp = sm + L.gp;
    const int tid = threadIdx.x;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const size_t hq = (size_t)bh * a.n;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += kThreads) gp[i] = pow_decay(log2g, (float)i);

    // reverse carries: the segment's workspace slot, or shared memory while it fits
    const size_t sidx = (size_t)bh * a.nseg + seg;
    float* Zg = a.ws + (RSUM ? a.ZhB : a.Zh_end) + sidx * D * DV;  // [D][DV]
    float* Sg = a.ws + (RSUM ? a.ShB : a.Sh_end) + sidx * D * D;    // [D][D]
    float* Zh = L.st_smem ? sm + L.Zh : Zg;
    float* Sh = L.st_smem ? sm + L.Sh : Sg;
    const int ldZ = L.st_smem ? ldV : DV;  // Zh rows: padded in shared memory
    if (RSUM) {
        for (int i = tid; i < D * DV; i += kThreads) Zh[(i / DV) * ldZ + i % DV] = 0.f;
        for (int i = tid; i < D * D; i += kThreads) Sh[i] = 0.f;
    } else {
        if (L.st_smem)
            for (int i = tid; i < D * DV; i += kThreads) Zh[(i / DV) * ldZ + i % DV] = Zg[i];
        // Sh + Sh^T, one thread per unordered pair (in place when it stays in the workspace)
        for (int e = tid; e < D * D; e += kThreads) {
            const int x = e / D, f = e - x * D;
            if (f < x) continue;
            const float s = Sg[x * D + f] + Sg[f * D + x];
            Sh[x * D + f] = s;
            Sh[f * D + x] = s;
        }
    }

    for (int c = c_end - 1; c >= c_begin; --c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        __syncthreads();  // the previous chunk's readers of the tiles and carries are done
        for (int i = tid; i < W * D; i += kThreads) {
            const int r = i / D, f = i - r * D;
            const bool in = r < Wc && HLA2_IN(row0 + r < a.n, 601);
            Qs[r * ldD + f] = in ? a.q[(hq + row0) * D + i] : 0.f;
            if (!RSUM) {
                const float kx = in ? a.k[(hq + row0) * D + i] : 0.f;
                Ks[r * ldD + f] = kx;
                Kt[f * ldW + r] = kx;
            }
        }
        for (int i = tid; i < W * DV; i += kThreads) {
            const int r = i / DV, x = i - r * DV;
            const bool in = r < Wc && HLA2_IN(row0 + r < a.n, 602);
            const float vx = in ? a.v[(hq + row0) * DV + i] : 0.f;
            Vt[x * ldW + r] = vx;
            if (!RSUM) Vs[r * ldV + x] = vx;
            Os[r * ldV + x] = in ? a.dout[(hq + row0) * DV + i] : 0.f;
        }
        const float* S0g = RSUM ? nullptr : a.chunk_states + ((size_t)bh * a.nchunks + c) * (size_t)(D * D + D * DV);
        const float* S0 = L.s0_smem ? sm + L.S0 : S0g;
        if (!RSUM) {  // S0 and Z0^T (the forward exports S0 [D][D] and Z0 [D][DV], row-major)
            if (L.s0_smem)
                for (int i = tid; i < (D * D) / 4; i += kThreads)
                    reinterpret_cast<float4*>(sm + L.S0)[i] = reinterpret_cast<const float4*>(S0g)[i];
            const float* Z0 = S0g + (size_t)D * D;
            for (int i = tid; i < D * DV; i += kThreads) {
                const int x = i / D, f = i - x * D;
                Z0t[x * ldD + f] = Z0[(size_t)f * DV + x];
            }
        }
        __syncthreads();

        // ---- D~ (and A~) -----------------------------------------------------------------
        tri_gram(Dt, ldW, Os, ldV, Vt, ldW, W, DV, gp, 2);
        if (!RSUM) tri_gram(At, ldW, Qs, ldD, Kt, ldW, W, D, gp, 1);
        __syncthreads();

        // ---- dP^T[f][j] = g^(2(Wc-1-j)) (Zh V^T)[f][j] + sum_{r >= j} q_r[f] D~[r][j] ---------
        simt::with_rm(D, W, [&](auto t) {
            constexpr int RM = decltype(t)::value;
            simt::for_blocks<RM>(D, W, [&](int m0, int n0) {
                simt::Acc<RM> acc;
                simt::zero(acc);
                simt::mac_r<RM>(acc, Zh + m0 * ldZ, ldZ, Vt + n0, ldW, DV);
                float cw[4];
#pragma unroll
                for (int b = 0; b < 4; ++b) cw[b] = n0 + b < Wc ? gp[2 * (Wc - 1 - n0 - b)] : 0.f;
#pragma unroll
                for (int i = 0; i < RM; ++i)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[i][b] *= cw[b];
                simt::mac_c<RM>(acc, Qs + m0, ldD, Dt + n0, ldW, n0, W);
#pragma unroll
                for (int i = 0; i < RM; ++i) {
                    simt::st4(dPt + (m0 + i) * ldW + n0, acc[i]);
                    if (!RSUM) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) dPs[(n0 + b) * ldD + m0 + i] = acc[i][b];
                    }
                }
            });
        });
        // ---- P = diag(g^(j+1)) Q S0 + A~ K -------------------------------------------------
        if (!RSUM) {
            simt::with_rm(W, D, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, D, [&](int m0, int n0) {
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, Qs + m0 * ldD, ldD, S0 + n0, D, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::scale_row(acc, i, gp[m0 + i + 1]);
                    simt::mac_r<RM>(acc, At + m0 * ldW, ldW, Ks + n0, ldD, min(W, m0 + RM));
#pragma unroll
                    for (int i = 0; i < RM; ++i) {
                        simt::st4(Ps + (m0 + i) * ldD + n0, acc[i]);
#pragma unroll
                        for (int b = 0; b < 4; ++b) Pt[(n0 + b) * ldW + m0 + i] = acc[i][b];
                    }
                });
            });
        }
        __syncthreads();

        if (!RSUM) {
            // ---- B~, dA~ ---------------------------------------------------------------------
            tri_gram(Bt, ldW, Qs, ldD, Pt, ldW, W, D, gp, 2);
            tri_gram(dAt, ldW, dPs, ldD, Kt, ldW, W, D, gp, 1);
            __syncthreads();

            // ---- dV, dQ, dK -> global ----------------------------------------------------------
            simt::with_rm(W, DV, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, DV, [&](int m0, int n0) {
                    if (m0 >= Wc) return;
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, Ps + m0 * ldD, ldD, Zh + n0, ldZ, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i)
                        simt::scale_row(acc, i, m0 + i < Wc ? gp[2 * (Wc - 1 - m0 - i)] : 0.f);
                    simt::mac_c<RM>(acc, Bt + m0, ldW, Os + n0, ldV, m0, W);
#pragma unroll
                    for (int i = 0; i < RM; ++i)
                        if (m0 + i < Wc && HLA2_IN(row0 + m0 + i < a.n, 603))
                            simt::st4(a.dv + (hq + row0 + m0 + i) * DV + n0, acc[i]);
                });
            });
            simt::with_rm(W, D, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, D, [&](int m0, int n0) {
                    if (m0 >= Wc) return;
                    const int kr = min(W, m0 + RM);
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, Os + m0 * ldV, ldV, Z0t + n0, ldD, DV);
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::scale_row(acc, i, gp[m0 + i + 1]);
                    simt::mac_r<RM>(acc, dPs + m0 * ldD, ldD, S0 + n0, D, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i) simt::scale_row(acc, i, gp[m0 + i + 1]);
                    simt::mac_r<RM>(acc, Dt + m0 * ldW, ldW, Ps + n0, ldD, kr);
                    simt::mac_r<RM>(acc, dAt + m0 * ldW, ldW, Ks + n0, ldD, kr);
#pragma unroll
                    for (int i = 0; i < RM; ++i)
                        if (m0 + i < Wc && HLA2_IN(row0 + m0 + i < a.n, 604))
                            simt::st4(a.dq + (hq + row0 + m0 + i) * D + n0, acc[i]);
                });
            });
            simt::with_rm(W, D, [&](auto t) {
                constexpr int RM = decltype(t)::value;
                simt::for_blocks<RM>(W, D, [&](int m0, int n0) {
                    if (m0 >= Wc) return;
                    simt::Acc<RM> acc;
                    simt::zero(acc);
                    simt::mac_r<RM>(acc, Ks + m0 * ldD, ldD, Sh + n0, D, D);
#pragma unroll
                    for (int i = 0; i < RM; ++i)
                        simt::scale_row(acc, i, m0 + i < Wc ? gp[Wc - 1 - m0 - i] : 0.f);
                    simt::mac_c<RM>(acc, At + m0, ldW, dPs + n0, ldD, m0, W);
                    simt::mac_c<RM>(acc, dAt + m0, ldW, Qs + n0, ldD, m0, W);
#pragma unroll
                    for (int i = 0; i < RM; ++i)
                        if (m0 + i < Wc && HLA2_IN(row0 + m0 + i < a.n, 605))
                            simt::st4(a.dk + (hq + row0 + m0 + i) * D + n0, acc[i]);
                });
            });
            __syncthreads();  // every read of the carries is done before they move
        }

        // ---- carries to the chunk start (each block owned by one thread) ---------------------
        const float rho = gp[Wc], rho2 = gp[2 * Wc];
        simt::with_rm(D, DV, [&](auto t) {
            constexpr int RM = decltype(t)::value;
            simt::for_blocks<RM>(D, DV, [&](int m0, int n0) {
                simt::Acc<RM> acc;
                simt::zero(acc);
                simt::mac_c<RM>(acc, Qs + m0, ldD, Os + n0, ldV, 0, Wc, [&](int r) { return gp[2 * (r + 1)]; });
#pragma unroll
                for (int i = 0; i < RM; ++i) simt::decay_add4(Zh + (m0 + i) * ldZ + n0, rho2, acc[i]);
            });
        });
        simt::with_rm(D, D, [&](auto t) {
            constexpr int RM = decltype(t)::value;
            simt::for_blocks<RM>(D, D, [&](int m0, int n0) {
                simt::Acc<RM> acc;
                simt::zero(acc);
                auto wj = [&](int j) { return gp[j + 1]; };
                simt::mac_r<RM>(acc, dPt + m0 * ldW, ldW, Qs + n0, ldD, Wc, wj);
                if (!RSUM) simt::mac_c<RM>(acc, Qs + m0, ldD, dPs + n0, ldD, 0, Wc, wj);
#pragma unroll
                for (int i = 0; i < RM; ++i) simt::decay_add4(Sh + (m0 + i) * D + n0, rho, acc[i]);
            });
        });
    }
    if (RSUM && L.st_smem) {
        __syncthreads();
        for (int i = tid; i < D * DV; i += kThreads) Zg[i] = Zh[(i / DV) * ldZ + i % DV];
        for (int i = tid; i < D * D; i += kThreads) Sg[i] = Sh[i];
    }
}

}  // namespace

size_t bwd_chunk_simt_smem(int d, int dv, int W) { return bs_layout(d, dv, W).total * sizeof(float); }

int launch_bwd_chunk_simt(const BwdArgsF& a, int d, int dv, bool rsum, cudaStream_t st) {
    if (a.nseg <= 0 || a.BH <= 0) return 0;
    if ((d & 15) || (dv & 15) || (a.W & 15)) return -1;
    const size_t smem = bwd_chunk_simt_smem(d, dv, a.W);
    auto kfn = rsum ? bwd_chunk_simt_kernel<true> : bwd_chunk_simt_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -1;
    kfn<<<dim3(a.nseg, a.BH), kThreads, smem, st>>>(a, d, dv);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(bwd_simt)
