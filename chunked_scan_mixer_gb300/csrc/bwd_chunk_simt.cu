// fp32 reverse-mode chunk kernel of the masked HLA-2 backward (SIMT): the same per-chunk
// algebra as the bf16 tensor-core kernel (bwd_chunk_mma.cuh), written as plain loops in
// float32 for float32 inputs of any d, dv in {16, 32, 64, 128}.  Gradients of the
// unnormalised output, equal to those of the serial recurrence (page "Higher-order Linear
// Attention", section summary §4.2: a reverse-mode scan reproduces the serial recurrence's
// gradients).  With p_t = S_t q_t, Z_t = g^2 Z_{t-1} + p_t v_t^T, o_t = q_t^T Z_t the
// adjoint is
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
// One CTA walks one segment's chunks from the last to the first.  The reverse carries live
// in the workspace (the segment's slot, updated in place); the forward states S0, Z0 come
// from the float32 state-export pass of the forward kernel.  RSUM mode starts from zero
// carries and keeps only what the reverse scan needs (D~, dP and the carry updates).
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kBsThreads = 256;

struct BsLayout {
    size_t Q, K, V, O, P, dP, At, Dt, Bt, dAt, gp, total;
};

__host__ __device__ inline BsLayout bs_layout(int D, int DV, int W) {
    BsLayout L;
    size_t o = 0;
    L.Q = o;   o += (size_t)W * D;
    L.K = o;   o += (size_t)W * D;
    L.V = o;   o += (size_t)W * DV;
    L.O = o;   o += (size_t)W * DV;
    L.P = o;   o += (size_t)W * D;
    L.dP = o;  o += (size_t)W * D;
    L.At = o;  o += (size_t)W * W;
    L.Dt = o;  o += (size_t)W * W;
    L.Bt = o;  o += (size_t)W * W;
    L.dAt = o; o += (size_t)W * W;
    L.gp = o;  o += 2 * (size_t)W + 2;
    L.total = o;
    return L;
}

template <bool RSUM>
__global__ void __launch_bounds__(kBsThreads) bwd_chunk_simt_kernel(const BwdArgsF a, int D, int DV) {
    extern __shared__ __align__(16) float sm[];
    const int W = a.W;
    const BsLayout L = bs_layout(D, DV, W);
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Vs = sm + L.V, *Os = sm + L.O, *Ps = sm + L.P, *dPs = sm + L.dP;
    float *At = sm + L.At, *Dt = sm + L.Dt, *Bt = sm + L.Bt, *dAt = sm + L.dAt, *gp = sm + L.gp;
    const int tid = threadIdx.x, NT = blockDim.x;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const size_t hq = (size_t)bh * a.n;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);

    const size_t sidx = (size_t)bh * a.nseg + seg;
    float* Zh = a.ws + (RSUM ? a.ZhB : a.Zh_end) + sidx * D * DV;  // [D][DV], updated in place
    float* Sh = a.ws + (RSUM ? a.ShB : a.Sh_end) + sidx * D * D;    // [D][D]
    if (RSUM) {
        for (int i = tid; i < D * DV; i += NT) Zh[i] = 0.f;
        for (int i = tid; i < D * D; i += NT) Sh[i] = 0.f;
    }

    for (int c = c_end - 1; c >= c_begin; --c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        __syncthreads();  // the previous chunk's readers of the tiles and carries are done
        for (int i = tid; i < W * D; i += NT) {
            const int r = i / D;
            const bool in = r < Wc && HLA2_IN(row0 + r < a.n, 601);
            Qs[i] = in ? a.q[(hq + row0) * D + i] : 0.f;
            if (!RSUM) Ks[i] = in ? a.k[(hq + row0) * D + i] : 0.f;
        }
        for (int i = tid; i < W * DV; i += NT) {
            const int r = i / DV;
            const bool in = r < Wc && HLA2_IN(row0 + r < a.n, 602);
            Vs[i] = in ? a.v[(hq + row0) * DV + i] : 0.f;
            Os[i] = in ? a.dout[(hq + row0) * DV + i] : 0.f;
        }
        const float* S0 = RSUM ? nullptr : a.chunk_states + ((size_t)bh * a.nchunks + c) * (size_t)(D * D + D * DV);
        const float* Z0 = RSUM ? nullptr : S0 + (size_t)D * D;
        __syncthreads();

        // ---- phase 1: D~ (and A~) ---------------------------------------------------------
        for (int e = tid; e < W * W; e += NT) {
            const int r = e / W, j = e % W;
            float sd = 0.f, sa = 0.f;
            if (j <= r) {
                for (int x = 0; x < DV; ++x) sd += Os[r * DV + x] * Vs[j * DV + x];
                if (!RSUM)
                    for (int x = 0; x < D; ++x) sa += Qs[r * D + x] * Ks[j * D + x];
            }
            Dt[e] = j <= r ? gp[2 * (r - j)] * sd : 0.f;
            if (!RSUM) At[e] = j <= r ? gp[r - j] * sa : 0.f;
        }
        __syncthreads();

        // ---- phase 2: dP (and P) -------------------------------------------------------------
        for (int e = tid; e < W * D; e += NT) {
            const int j = e / D, f = e % D;
            float s0 = 0.f, s1 = 0.f;
            if (j < Wc)
                for (int x = 0; x < DV; ++x) s0 += Vs[j * DV + x] * Zh[(size_t)f * DV + x];
            for (int r = j; r < W; ++r) s1 += Dt[r * W + j] * Qs[r * D + f];
            dPs[e] = (j < Wc ? gp[2 * (Wc - 1 - j)] * s0 : 0.f) + s1;
            if (!RSUM) {
                float p0 = 0.f, p1 = 0.f;
                for (int x = 0; x < D; ++x) p0 += Qs[j * D + x] * S0[(size_t)x * D + f];
                for (int i = 0; i <= j; ++i) p1 += At[j * W + i] * Ks[i * D + f];
                Ps[e] = gp[j + 1] * p0 + p1;
            }
        }
        __syncthreads();

        if (!RSUM) {
            // ---- phase 3: B~, dA~ ----------------------------------------------------------------
            for (int e = tid; e < W * W; e += NT) {
                const int r = e / W, j = e % W;
                float sb = 0.f, sa = 0.f;
                if (j <= r)
                    for (int x = 0; x < D; ++x) {
                        sb += Qs[r * D + x] * Ps[j * D + x];
                        sa += dPs[r * D + x] * Ks[j * D + x];
                    }
                Bt[e] = j <= r ? gp[2 * (r - j)] * sb : 0.f;
                dAt[e] = j <= r ? gp[r - j] * sa : 0.f;
            }
            __syncthreads();

            // ---- phase 4: dV, dQ, dK -> global ---------------------------------------------------
            for (int e = tid; e < Wc * DV; e += NT) {
                const int j = e / DV, x = e % DV;
                float s0 = 0.f, s1 = 0.f;
                for (int f = 0; f < D; ++f) s0 += Ps[j * D + f] * Zh[(size_t)f * DV + x];
                for (int r = j; r < Wc; ++r) s1 += Bt[r * W + j] * Os[r * DV + x];
                if (HLA2_IN(row0 + j < a.n, 603)) a.dv[(hq + row0) * DV + e] = gp[2 * (Wc - 1 - j)] * s0 + s1;
            }
            for (int e = tid; e < Wc * D; e += NT) {
                const int r = e / D, f = e % D;
                float sz = 0.f, ss = 0.f, sp = 0.f;
                for (int x = 0; x < DV; ++x) sz += Os[r * DV + x] * Z0[(size_t)f * DV + x];
                for (int x = 0; x < D; ++x) ss += dPs[r * D + x] * S0[(size_t)x * D + f];
                for (int j = 0; j <= r; ++j) sp += Dt[r * W + j] * Ps[j * D + f] + dAt[r * W + j] * Ks[j * D + f];
                if (HLA2_IN(row0 + r < a.n, 604)) a.dq[(hq + row0) * D + e] = gp[r + 1] * (gp[r + 1] * sz + ss) + sp;
            }
            for (int e = tid; e < Wc * D; e += NT) {
                const int i = e / D, f = e % D;
                float sh = 0.f, sr = 0.f;
                for (int x = 0; x < D; ++x) sh += Ks[i * D + x] * (Sh[(size_t)x * D + f] + Sh[(size_t)f * D + x]);
                for (int r = i; r < Wc; ++r) sr += At[r * W + i] * dPs[r * D + f] + dAt[r * W + i] * Qs[r * D + f];
                if (HLA2_IN(row0 + i < a.n, 605)) a.dk[(hq + row0) * D + e] = gp[Wc - 1 - i] * sh + sr;
            }
            __syncthreads();  // every read of the carries is done before they move
        }

        // ---- carries to the chunk start (each element owned by one thread) -----------------
        const float rho = gp[Wc], rho2 = gp[2 * Wc];
        for (int e = tid; e < D * DV; e += NT) {
            const int f = e / DV, x = e % DV;
            float s = 0.f;
            for (int r = 0; r < Wc; ++r) s += gp[2 * (r + 1)] * Qs[r * D + f] * Os[r * DV + x];
            Zh[e] = rho2 * Zh[e] + s;
        }
        for (int e = tid; e < D * D; e += NT) {
            const int f = e / D, x = e % D;
            float s = 0.f;
            for (int j = 0; j < Wc; ++j) s += gp[j + 1] * dPs[j * D + f] * Qs[j * D + x];
            Sh[e] = rho * Sh[e] + s;
        }
    }
}

}  // namespace

size_t bwd_chunk_simt_smem(int d, int dv, int W) { return bs_layout(d, dv, W).total * sizeof(float); }

int launch_bwd_chunk_simt(const BwdArgsF& a, int d, int dv, bool rsum, cudaStream_t st) {
    if (a.nseg <= 0 || a.BH <= 0) return 0;
    const size_t smem = bwd_chunk_simt_smem(d, dv, a.W);
    auto kfn = rsum ? bwd_chunk_simt_kernel<true> : bwd_chunk_simt_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -1;
    kfn<<<dim3(a.nseg, a.BH), kBsThreads, smem, st>>>(a, d, dv);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2

HLA2_DEBUG_READER(bwd_simt)
