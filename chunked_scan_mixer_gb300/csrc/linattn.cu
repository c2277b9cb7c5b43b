// Masked first-order linear attention, chunk-parallel (float32 arithmetic, SIMT):
//     u_t = sum_{l <= t} g^(t-l) (q_t . k_l) v_l = P_t^T q_t,   P_t = g P_{t-1} + k_t v_t^T.
// It is the inner pass of the masked third-order output (page "Higher-order Linear
// Attention", technical summary item "3. Dritte Ordnung HLA"): with every factor of
// A A^T A causally masked, the third-order output is the masked second-order output whose
// values are these u_t, so the library evaluates it as this pass followed by the
// second-order forward.
//
// Per chunk of width W (rows r, P0 the state at the chunk start):
//   U = diag(g^(r+1)) Q P0 + ((Q K^T) * [l <= r] g^(r-l)) V,   P <- g^Wc P0 + K~^T V,
// with K~ = diag(g^(Wc-1-l)) K.  Segments of chunks run one CTA each: a summary pass stores
// each segment's P (from zero), a decayed prefix over the segments gives the carries, and
// the output pass starts every segment from its carry.
#include "kernels.h"

namespace hla2 {

namespace {

constexpr int kLaThreads = 256;

struct LaSmem {
    size_t Q, K, V, A, P, gp, total;
};

__host__ __device__ inline LaSmem la_smem(int D, int DV, int W) {
    LaSmem L;
    size_t o = 0;
    L.Q = o;  o += (size_t)W * D;
    L.K = o;  o += (size_t)W * D;
    L.V = o;  o += (size_t)W * DV;
    L.A = o;  o += (size_t)W * W;
    L.P = o;  o += (size_t)D * DV;
    L.gp = o; o += (size_t)W + 1;
    L.total = o;
    return L;
}

template <typename T, bool SUMMARY>
__global__ void __launch_bounds__(kLaThreads) la_chunk_kernel(const LaArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int D = a.d, DV = a.dv, W = a.W;
    const LaSmem L = la_smem(D, DV, W);
    float *Qs = sm + L.Q, *Ks = sm + L.K, *Vs = sm + L.V, *As = sm + L.A, *P = sm + L.P, *gp = sm + L.gp;
    const int tid = threadIdx.x, NT = blockDim.x;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const T* q = static_cast<const T*>(a.q) + (size_t)bh * a.n * D;
    const T* k = static_cast<const T*>(a.k) + (size_t)bh * a.n * D;
    const T* v = static_cast<const T*>(a.v) + (size_t)bh * a.n * DV;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i <= W; i += NT) gp[i] = pow_decay(log2g, (float)i);
    const size_t ddv = (size_t)D * DV;
    for (int i = tid; i < D * DV; i += NT)
        P[i] = SUMMARY ? 0.f : a.ws[a.Pin + ((size_t)bh * a.nseg + seg) * ddv + i];

    for (int c = c_begin; c < c_end; ++c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        __syncthreads();
        for (int i = tid; i < W * D; i += NT) {
            const bool ok = i / D < Wc;
            Qs[i] = ok ? to_f32(q[(size_t)row0 * D + i]) : 0.f;
            Ks[i] = ok ? to_f32(k[(size_t)row0 * D + i]) : 0.f;
        }
        for (int i = tid; i < W * DV; i += NT) Vs[i] = i / DV < Wc ? to_f32(v[(size_t)row0 * DV + i]) : 0.f;
        __syncthreads();
        if (!SUMMARY) {
            for (int e = tid; e < W * W; e += NT) {
                const int r = e / W, l = e % W;
                float s = 0.f;
                if (l <= r)
                    for (int f = 0; f < D; ++f) s += Qs[r * D + f] * Ks[l * D + f];
                As[e] = l <= r ? gp[r - l] * s : 0.f;
            }
            __syncthreads();
            T* out = static_cast<T*>(a.u) + ((size_t)bh * a.n + row0) * DV;
            for (int e = tid; e < Wc * DV; e += NT) {
                const int r = e / DV, x = e % DV;
                float s0 = 0.f, s1 = 0.f;
                for (int f = 0; f < D; ++f) s0 += Qs[r * D + f] * P[f * DV + x];
                for (int l = 0; l <= r; ++l) s1 += As[r * W + l] * Vs[l * DV + x];
                out[e] = from_f32<T>(gp[r + 1] * s0 + s1);
            }
            __syncthreads();  // P is read above and updated below
        }
        const float rho = gp[Wc];
        for (int e = tid; e < D * DV; e += NT) {
            const int f = e / DV, x = e % DV;
            float s = 0.f;
            for (int l = 0; l < Wc; ++l) s += gp[Wc - 1 - l] * Ks[l * D + f] * Vs[l * DV + x];
            P[e] = rho * P[e] + s;
        }
    }
    if (SUMMARY || (a.final_P && seg == a.nseg - 1)) {
        __syncthreads();
        float* dst = SUMMARY ? a.ws + a.PB + ((size_t)bh * (a.nseg - 1) + seg) * ddv : a.final_P + (size_t)bh * ddv;
        for (int i = tid; i < D * DV; i += NT) dst[i] = P[i];
    }
}

// One CTA per head: S, P copied; Y = S C - G (the second-order Z on values u); m = the unit
// pass's P column 0 (sum of keys); y = (S C1 - G1) column 0 (Z on the unit values).
__global__ void __launch_bounds__(kLaThreads)
    hla3_assemble_kernel(float* fin, const float* pk_num, const float* pk_den, const float* p_num, const float* p_den,
                         int d, int dv, int w) {
    const size_t head = blockIdx.x;
    const size_t sf = (size_t)d * d + 2 * (size_t)d * dv + 2 * (size_t)d;
    const size_t sw = (size_t)d * d + 2 * (size_t)d * w + 2 * (size_t)d;
    float* o = fin + head * sf;
    const float* S = pk_num + head * sf;
    const float* C = S + (size_t)d * d;
    const float* G = C + (size_t)d * dv;
    const float* C1 = pk_den + head * sw + (size_t)d * d;
    const float* G1 = C1 + (size_t)d * w;
    for (int i = threadIdx.x; i < d * d; i += kLaThreads) o[i] = S[i];
    for (int i = threadIdx.x; i < d * dv; i += kLaThreads) {
        o[(size_t)d * d + i] = p_num[head * d * dv + i];
        const int a = i / dv, x = i % dv;
        float s = 0.f;
        for (int j = 0; j < d; ++j) s += S[(size_t)a * d + j] * C[(size_t)j * dv + x];
        o[(size_t)d * d + (size_t)d * dv + i] = s - G[i];
    }
    for (int a = threadIdx.x; a < d; a += kLaThreads) {
        float s = 0.f;
        for (int j = 0; j < d; ++j) s += S[(size_t)a * d + j] * C1[(size_t)j * w];
        o[(size_t)d * d + 2 * (size_t)d * dv + a] = p_den[head * d * w + (size_t)a * w];
        o[(size_t)d * d + 2 * (size_t)d * dv + d + a] = s - G1[(size_t)a * w];
    }
}

__global__ void __launch_bounds__(kLaThreads) la_init_kernel(const LaArgs a) {
    const size_t ddv = (size_t)a.d * a.dv;
    float* dst = a.ws + a.Pin + (size_t)blockIdx.x * a.nseg * ddv;
    for (size_t i = threadIdx.x; i < ddv; i += kLaThreads) dst[i] = 0.f;
}

template <typename T>
int la_pass(const LaArgs& a, bool summary, int count, cudaStream_t st) {
    if (count <= 0) return 0;
    const size_t smem = la_smem(a.d, a.dv, a.W).total * sizeof(float);
    auto kfn = summary ? la_chunk_kernel<T, true> : la_chunk_kernel<T, false>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
    kfn<<<dim3(count, a.BH), kLaThreads, smem, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <typename T>
__global__ void __launch_bounds__(kLaThreads) unit_rows_kernel(T* e0, size_t count, int w) {
    const size_t i = (size_t)blockIdx.x * kLaThreads + threadIdx.x;
    if (i < count) e0[i] = from_f32<T>((i % (size_t)w) == 0 ? 1.f : 0.f);
}

template <typename T>
__global__ void __launch_bounds__(kLaThreads) divide_rows_kernel(T* out, const T* den, size_t count, int dv, int w,
                                                                 float eps) {
    const size_t i = (size_t)blockIdx.x * kLaThreads + threadIdx.x;
    if (i >= count) return;
    const size_t row = i / (size_t)dv;
    out[i] = from_f32<T>(to_f32(out[i]) / (to_f32(den[row * w]) + eps));
}

unsigned blocks(size_t n) { return (unsigned)((n + kLaThreads - 1) / kLaThreads); }

}  // namespace

size_t first_order_smem(int d, int dv, int W) { return la_smem(d, dv, W).total * sizeof(float); }

int launch_hla3_assemble_state(float* fin, const float* pk_num, const float* pk_den, const float* p_num,
                               const float* p_den, long heads, int d, int dv, int w, cudaStream_t st) {
    if (heads <= 0) return 0;
    hla3_assemble_kernel<<<(unsigned)heads, kLaThreads, 0, st>>>(fin, pk_num, pk_den, p_num, p_den, d, dv, w);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_unit_rows(void* e0, size_t rows, int w, bool is_bf16, cudaStream_t st) {
    const size_t c = rows * (size_t)w;
    if (c == 0) return 0;
    if (is_bf16)
        unit_rows_kernel<bf16><<<blocks(c), kLaThreads, 0, st>>>(static_cast<bf16*>(e0), c, w);
    else
        unit_rows_kernel<float><<<blocks(c), kLaThreads, 0, st>>>(static_cast<float*>(e0), c, w);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_divide_rows(void* out, const void* den, size_t rows, int dv, int w, float eps, bool is_bf16,
                       cudaStream_t st) {
    const size_t c = rows * (size_t)dv;
    if (c == 0) return 0;
    if (is_bf16)
        divide_rows_kernel<bf16><<<blocks(c), kLaThreads, 0, st>>>(static_cast<bf16*>(out),
                                                                   static_cast<const bf16*>(den), c, dv, w, eps);
    else
        divide_rows_kernel<float><<<blocks(c), kLaThreads, 0, st>>>(static_cast<float*>(out),
                                                                    static_cast<const float*>(den), c, dv, w, eps);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_first_order_forward(const LaArgs& a, bool is_bf16, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    la_init_kernel<<<a.BH, kLaThreads, 0, st>>>(a);
    if (cudaPeekAtLastError() != cudaSuccess) return -1;
    LaArgs b = a;
    b.seg0 = 0;
    if (a.nseg > 1) {
        if (is_bf16 ? la_pass<bf16>(b, true, a.nseg - 1, st) : la_pass<float>(b, true, a.nseg - 1, st)) return -1;
        const size_t ddv = (size_t)a.d * a.dv;
        if (launch_linear_scan(a.ws + a.PB, a.ws + a.Pin, a.BH, a.H, a.nseg - 1, ddv, (size_t)(a.nseg - 1) * ddv,
                               (size_t)a.nseg * ddv, true, a.gamma, a.seg_chunks * a.W, 1, st))
            return -1;
    }
    return is_bf16 ? la_pass<bf16>(b, false, a.nseg, st) : la_pass<float>(b, false, a.nseg, st);
}

}  // namespace hla2
