// Asymmetric Higher-order Linear Attention (AHLA), chunk-parallel forward (page
// "Higher-order Linear Attention": technical summary item "2. Asymmetrische Lineare
// Aufmerksamkeit hoeherer Ordnung (AHLA)", the operator Q (K^T Q)(K^T V) with streaming
// summaries P^KV, m^K, E, n; section summary §6.1 masked streaming identity, §6.2
// chunk-parallel scan, §6.3 decay and normalisation).
//
// Per head and token (pairs i <= j <= t, weight g^(t-i)):
//   P_t = g P_{t-1} + k_t v_t^T,   E_t = g E_{t-1} + k_t (q_t^T P_t),   o_t = q_t^T E_t,
//   m_t = g m_{t-1} + k_t,         n_t = g n_{t-1} + k_t (q_t . m_t),   den_t = q_t . n_t.
// Per chunk (rows r, carries P0, E0, m0, n0 at the chunk start) both cascaded products use
// the same masked matrix A~[r, j] = [j <= r] g^(r-j) (q_r . k_j):
//   Inner = diag(g^(r+1)) Q P0 + A~ V,           O   = diag(g^(r+1)) Q E0 + A~ Inner,
//   idn   = g^(r+1) Q m0 + A~ 1,                 den = g^(r+1) Q n0 + A~ idn,
//   P <- g^Wc P0 + K~^T V,  E <- g^Wc E0 + K~^T Inner,  K~ = diag(g^(Wc-1-i)) K  (m, n alike).
// Segment summaries add R = sum_j k_j q_j^T (undecayed: a cross pair's decay telescopes to the
// later segment's attenuation), and segments combine, A earlier, rho = g^len(B), as
//   P = rho P_A + P_B,  E = rho E_A + E_B + rho R_B P_A  (m, n with P -> m).
// So the carry scan is a decayed prefix of P, independent products X_s = E_B[s] +
// rho R_B[s] P_in[s], and a decayed prefix of X.
//
// bf16 inputs and outputs, fp32 state, d == dv in {16, 32, 64, 128}, chunk 32 or 64, legacy
// tensor cores (mma.m16n8k16) with the per-warp tile helpers of common.cuh.
#include "kernels.h"

namespace hla2 {

namespace {

template <int D, int W>
struct AhlaCfg {
    static constexpr int DV = D;
    static constexpr int NW = D <= 32 ? 4 : (D == 64 ? 8 : 16);
    static constexpr int NT = NW * 32;
    static constexpr int LD = D + 8, LW = W + 8;
    static constexpr int TW = W / 16, TD = D / 16;
    static constexpr int TILES = TD * TD;                       // d x d (and d x dv) state tiles
    static constexpr int PER = (TILES + NW - 1) / NW;
    static constexpr size_t ROWS = (size_t)W * LD * 2;           // one [W][D] bf16 tile
    static constexpr size_t oQ = 0, oK = ROWS, oV = 2 * ROWS, oKt = 3 * ROWS, oIn = 4 * ROWS;
    static constexpr size_t oAB = 5 * ROWS;
    static constexpr size_t oP = oAB + (size_t)W * LW * 2;       // [D][D] bf16
    static constexpr size_t oE = oP + (size_t)D * LD * 2;
    static constexpr size_t oF = oE + (size_t)D * LD * 2;         // floats
    // gp[2W+2] | qm[W] | qn[W] | idn[W] | den[W] | m[D] | n[D]
    static constexpr size_t nF = (2 * W + 2) + 4 * W + 2 * D;
    static constexpr size_t BYTES = oF + ((nF * 4 + 15) / 16) * 16;
};

template <int D, int W, bool SUMMARY>
__global__ void __launch_bounds__(AhlaCfg<D, W>::NT) ahla_chunk_kernel(const AhlaArgs a) {
    using Cfg = AhlaCfg<D, W>;
    constexpr int DV = D, NW = Cfg::NW, NT = Cfg::NT, LD = Cfg::LD, LW = Cfg::LW, TW = Cfg::TW, TD = Cfg::TD;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16* Qs = reinterpret_cast<bf16*>(smem + Cfg::oQ);
    bf16* Ks = reinterpret_cast<bf16*>(smem + Cfg::oK);
    bf16* Vs = reinterpret_cast<bf16*>(smem + Cfg::oV);
    bf16* Kt = reinterpret_cast<bf16*>(smem + Cfg::oKt);
    bf16* In = reinterpret_cast<bf16*>(smem + Cfg::oIn);
    bf16* AB = reinterpret_cast<bf16*>(smem + Cfg::oAB);
    bf16* Pst = reinterpret_cast<bf16*>(smem + Cfg::oP);
    bf16* Est = reinterpret_cast<bf16*>(smem + Cfg::oE);
    float* gp = reinterpret_cast<float*>(smem + Cfg::oF);
    float* qm = gp + 2 * W + 2;
    float* qn = qm + W;
    float* idn = qn + W;
    float* den = idn + W;
    float* ms = den + W;
    float* ns = ms + D;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const bf16* q = static_cast<const bf16*>(a.q) + (size_t)bh * a.n * D;
    const bf16* k = static_cast<const bf16*>(a.k) + (size_t)bh * a.n * D;
    const bf16* v = static_cast<const bf16*>(a.v) + (size_t)bh * a.n * DV;
    const bool norm = a.normalize != 0;
    // the denominator's summaries m, n are carried when the output is normalised or the
    // final state is asked for
    const bool track = norm || a.final_state != nullptr;

    const float g = head_decay(a.gamma, bh, a.H);
    const float log2g = log2f(g);
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);

    // fp32 state tiles owned per warp: P, E (d x dv) and, for summaries, R (d x d)
    float Pacc[Cfg::PER][2][4], Eacc[Cfg::PER][2][4], Racc[SUMMARY ? Cfg::PER : 1][2][4];
    const size_t cidx = (size_t)bh * a.nseg + seg;
#pragma unroll
    for (int s = 0; s < Cfg::PER; ++s) {
        const int t = warp + s * NW;
        const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const size_t e = (size_t)acc_row(m0, i) * DV + acc_col(n0, h, i);
                const bool ok = !SUMMARY && t < Cfg::TILES;
                Pacc[s][h][i] = ok ? a.ws[a.L.Pin + cidx * D * DV + e] : 0.f;
                Eacc[s][h][i] = ok ? a.ws[a.L.Ein + cidx * D * DV + e] : 0.f;
                if (SUMMARY) Racc[s][h][i] = 0.f;
            }
    }
    for (int f = tid; f < D; f += NT) {
        ms[f] = SUMMARY ? 0.f : a.ws[a.L.min + cidx * D + f];
        ns[f] = SUMMARY ? 0.f : a.ws[a.L.nin + cidx * D + f];
    }

    auto publish_state = [&]() {
#pragma unroll
        for (int s = 0; s < Cfg::PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int r = acc_row(m0, i), c = acc_col(n0, h, i);
                    *reinterpret_cast<uint32_t*>(&Pst[r * LD + c]) = pack_bf16x2(Pacc[s][h][i], Pacc[s][h][i + 1]);
                    *reinterpret_cast<uint32_t*>(&Est[r * LD + c]) = pack_bf16x2(Eacc[s][h][i], Eacc[s][h][i + 1]);
                }
        }
    };
    publish_state();

    auto load_chunk = [&](int c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        constexpr int CPR = D / 8;
        for (int i = tid; i < W * CPR; i += NT) {
            const int r = i / CPR, p = (i % CPR) * 8;
            if (r < Wc) {
                cp_async16(&Qs[r * LD + p], q + (size_t)(row0 + r) * D + p);
                cp_async16(&Ks[r * LD + p], k + (size_t)(row0 + r) * D + p);
                cp_async16(&Vs[r * LD + p], v + (size_t)(row0 + r) * DV + p);
            } else {
                *reinterpret_cast<uint4*>(&Qs[r * LD + p]) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(&Ks[r * LD + p]) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(&Vs[r * LD + p]) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_commit();
    };
    if (c_begin < c_end) load_chunk(c_begin);

    for (int c = c_begin; c < c_end; ++c) {
        const int Wc = min(W, a.n - c * W);
        cp_async_wait_all();
        __syncthreads();

        // ---- K~ rows; the denominator's carry reads q . m0, q . n0 ----------------------
        for (int i = tid; i < W * D; i += NT) {
            const int r = i / D, f = i % D;
            Kt[r * LD + f] = from_f32<bf16>((r < Wc ? gp[Wc - 1 - r] : 0.f) * to_f32(Ks[r * LD + f]));
        }
        if (track) {
            for (int r = tid; r < W; r += NT) {
                float sm = 0.f, sn = 0.f;
                for (int f = 0; f < D; ++f) {
                    const float qf = to_f32(Qs[r * LD + f]);
                    sm += qf * ms[f];
                    sn += qf * ns[f];
                }
                qm[r] = sm;
                qn[r] = sn;
            }
        }
        __syncthreads();

        // ---- A~ = mask(Q K^T) * g^(r-j) ----------------------------------------------------
        for (int t = warp; t < TW * TW; t += NW) {
            const int rb = t / TW, cb = t % TW;
            if (cb > rb) continue;
            float acc[2][4];
            zero_acc(acc);
            warp_tile_mma<false, false>(acc, Qs, LD, rb * 16, Ks, LD, cb * 16, 0, D);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int r = acc_row(rb * 16, i), col = acc_col(cb * 16, h, i);
                    const float v0 = col <= r ? gp[r - col] * acc[h][i] : 0.f;
                    const float v1 = col + 1 <= r ? gp[r - col - 1] * acc[h][i + 1] : 0.f;
                    *reinterpret_cast<uint32_t*>(&AB[r * LW + col]) = pack_bf16x2(v0, v1);
                }
        }
        __syncthreads();
        // tiles above the diagonal block row are never read: products stop at (rb + 1) * 16
        if (track) {  // idn = g^(r+1) q.m0 + row sums of A~
            for (int r = tid; r < W; r += NT) {
                float s = 0.f;
                for (int j = 0; j <= r; ++j) s += to_f32(AB[r * LW + j]);
                idn[r] = r < Wc ? gp[r + 1] * qm[r] + s : 0.f;
            }
        }

        // ---- Inner = diag(g^(r+1)) Q P0 + A~ V ----------------------------------------------
        for (int t = warp; t < TW * TD; t += NW) {
            const int rb = t / TD, eb = t % TD;
            float acc[2][4];
            zero_acc(acc);
            warp_tile_mma<false, true>(acc, Qs, LD, rb * 16, Pst, LD, eb * 16, 0, D);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
            warp_tile_mma<false, true>(acc, AB, LW, rb * 16, Vs, LD, eb * 16, 0, (rb + 1) * 16);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int r = acc_row(rb * 16, i), col = acc_col(eb * 16, h, i);
                    *reinterpret_cast<uint32_t*>(&In[r * LD + col]) =
                        r < Wc ? pack_bf16x2(acc[h][i], acc[h][i + 1]) : 0u;
                }
        }
        __syncthreads();

        if (!SUMMARY) {
            if (norm) {  // den = g^(r+1) q.n0 + A~ idn
                for (int r = tid; r < W; r += NT) {
                    float s = 0.f;
                    for (int j = 0; j <= r; ++j) s += to_f32(AB[r * LW + j]) * idn[j];
                    den[r] = gp[r + 1] * qn[r] + s;
                }
                __syncthreads();
            }
            // ---- O = diag(g^(r+1)) Q E0 + A~ Inner -> out ----------------------------------
            bf16* outp = static_cast<bf16*>(a.out) + ((size_t)bh * a.n + (size_t)c * W) * DV;
            for (int t = warp; t < TW * TD; t += NW) {
                const int rb = t / TD, eb = t % TD;
                float acc[2][4];
                zero_acc(acc);
                warp_tile_mma<false, true>(acc, Qs, LD, rb * 16, Est, LD, eb * 16, 0, D);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
                warp_tile_mma<false, true>(acc, AB, LW, rb * 16, In, LD, eb * 16, 0, (rb + 1) * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(eb * 16, h, i);
                        if (r >= Wc) continue;
                        float o0 = acc[h][i], o1 = acc[h][i + 1];
                        if (norm) {
                            const float inv = 1.f / (den[r] + a.eps);
                            o0 *= inv;
                            o1 *= inv;
                        }
                        *reinterpret_cast<uint32_t*>(&outp[(size_t)r * DV + col]) = pack_bf16x2(o0, o1);
                    }
            }
        }

        // ---- state: P <- g^Wc P0 + K~^T V, E <- g^Wc E0 + K~^T Inner (R += K^T Q) ------------
        const float rho = gp[Wc];
#pragma unroll
        for (int s = 0; s < Cfg::PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    Pacc[s][h][i] *= rho;
                    Eacc[s][h][i] *= rho;
                }
            warp_tile_mma<true, true>(Pacc[s], Kt, LD, m0, Vs, LD, n0, 0, W);
            warp_tile_mma<true, true>(Eacc[s], Kt, LD, m0, In, LD, n0, 0, W);
            if (SUMMARY) warp_tile_mma<true, true>(Racc[s], Ks, LD, m0, Qs, LD, n0, 0, W);
        }
        for (int f = tid; f < D; f += NT) {
            float sm = 0.f, sn = 0.f;
            for (int r = 0; r < Wc; ++r) {
                const float kf = to_f32(Kt[r * LD + f]);
                sm += kf;
                if (track) sn += kf * idn[r];
            }
            ms[f] = rho * ms[f] + sm;
            ns[f] = rho * ns[f] + sn;
        }
        __syncthreads();  // every read of the chunk tiles, Pst and Est is done
        publish_state();
        if (c + 1 < c_end) load_chunk(c + 1);
    }
    __syncthreads();

    if (!SUMMARY && a.final_state && seg == a.nseg - 1) {  // state after token n: P | E | m | n
        float* fs = a.final_state + (size_t)bh * (2 * D * DV + 2 * D);
#pragma unroll
        for (int s = 0; s < Cfg::PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const size_t e = (size_t)acc_row(m0, i) * DV + acc_col(n0, h, i);
                    *reinterpret_cast<float2*>(&fs[e]) = make_float2(Pacc[s][h][i], Pacc[s][h][i + 1]);
                    *reinterpret_cast<float2*>(&fs[D * DV + e]) = make_float2(Eacc[s][h][i], Eacc[s][h][i + 1]);
                }
        }
        for (int f = tid; f < D; f += NT) {
            fs[2 * D * DV + f] = ms[f];
            fs[2 * D * DV + D + f] = ns[f];
        }
    }
    if (SUMMARY) {
        const size_t si = (size_t)bh * a.nsum + seg;
        float* dP = a.ws + a.L.PB + si * D * DV;
        float* dE = a.ws + a.L.EB + si * D * DV;
        float* dR = a.ws + a.L.RB + si * D * D;
#pragma unroll
        for (int s = 0; s < Cfg::PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const size_t e = (size_t)acc_row(m0, i) * DV + acc_col(n0, h, i);
                    *reinterpret_cast<float2*>(&dP[e]) = make_float2(Pacc[s][h][i], Pacc[s][h][i + 1]);
                    *reinterpret_cast<float2*>(&dE[e]) = make_float2(Eacc[s][h][i], Eacc[s][h][i + 1]);
                    *reinterpret_cast<float2*>(&dR[e]) = make_float2(Racc[s][h][i], Racc[s][h][i + 1]);
                }
        }
        for (int f = tid; f < D; f += NT) {
            a.ws[a.L.mB + si * D + f] = ms[f];
            a.ws[a.L.nB + si * D + f] = ns[f];
        }
    }
    (void)lane;
}

constexpr int kScanThreads = 256;

// Carries into segment 0: the initial state [P | E | m | n] (zero without one); clears the
// status word.  The scans then seed every later carry from these.
__global__ void __launch_bounds__(kScanThreads) ahla_init_kernel(const AhlaArgs a, int D) {
    const int bh = blockIdx.x, tid = threadIdx.x;
    if (bh == 0 && tid == 0) *reinterpret_cast<int*>(a.ws) = 0;
    const size_t c0 = (size_t)bh * a.nseg;
    const float* init = a.init_state ? a.init_state + (size_t)bh * ahla_state_floats(D, D) : nullptr;
    for (int i = tid; i < D * D; i += kScanThreads) {
        a.ws[a.L.Pin + c0 * D * D + i] = init ? init[i] : 0.f;
        a.ws[a.L.Ein + c0 * D * D + i] = init ? init[(size_t)D * D + i] : 0.f;
    }
    for (int i = tid; i < D; i += kScanThreads) {
        a.ws[a.L.min + c0 * D + i] = init ? init[2 * (size_t)D * D + i] : 0.f;
        a.ws[a.L.nin + c0 * D + i] = init ? init[2 * (size_t)D * D + D + i] : 0.f;
    }
}

// X_s = E_B[s] + rho R_B[s] P_in[s] and Xn_s = n_B[s] + rho R_B[s] m_in[s], in place
// (256 threads in a 16 x 16 grid, register tiles as in the symmetric scan's cross kernel).
template <int TM>
__global__ void __launch_bounds__(kScanThreads) ahla_cross_kernel(const AhlaArgs a, int seg_tokens) {
    constexpr int D = 16 * TM, TN = TM;
    extern __shared__ __align__(16) float sm[];
    float* Rs = sm;            // D x D
    float* Ps = Rs + D * D;    // D x D
    float* mv = Ps + D * D;    // D
    const int s = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const size_t sb = (size_t)bh * a.nsum + s, si = (size_t)bh * a.nseg + s;
    const float* R = a.ws + a.L.RB + sb * D * D;
    const float* P = a.ws + a.L.Pin + si * D * D;
    for (int i = tid; i < D * D / 4; i += kScanThreads) {
        reinterpret_cast<float4*>(Rs)[i] = reinterpret_cast<const float4*>(R)[i];
        reinterpret_cast<float4*>(Ps)[i] = reinterpret_cast<const float4*>(P)[i];
    }
    for (int i = tid; i < D; i += kScanThreads) mv[i] = a.ws[a.L.min + si * D + i];
    __syncthreads();
    const float rho = pow_decay(log2f(head_decay(a.gamma, bh, a.H)), (float)seg_tokens);
    const int tr = tid / 16, tc0 = (tid % 16) * TN;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int x = 0; x < D; ++x) {
        float av[TM], bv[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) av[i] = Rs[(tr + 16 * i) * D + x];
#pragma unroll
        for (int j = 0; j < TN; ++j) bv[j] = Ps[x * D + tc0 + j];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] += av[i] * bv[j];
    }
    float* E = a.ws + a.L.EB + sb * D * D;
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) E[(size_t)(tr + 16 * i) * D + tc0 + j] += rho * acc[i][j];
    if (a.normalize || a.final_state) {
        float* nb = a.ws + a.L.nB + sb * D;
        for (int r = tid; r < D; r += kScanThreads) {
            float t = 0.f;
            for (int x = 0; x < D; ++x) t += Rs[r * D + x] * mv[x];
            nb[r] += rho * t;
        }
    }
}

template <int D, int W>
int launch_chunk_t(const AhlaArgs& a, bool summary, cudaStream_t st) {
    using Cfg = AhlaCfg<D, W>;
    auto kfn = summary ? ahla_chunk_kernel<D, W, true> : ahla_chunk_kernel<D, W, false>;
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::BYTES) != cudaSuccess)
        return -1;
    kfn<<<dim3(a.nseg_launch, a.BH), Cfg::NT, Cfg::BYTES, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int TM>
int launch_cross_t(const AhlaArgs& a, cudaStream_t st) {
    constexpr int D = 16 * TM;
    const size_t smem = (size_t)(2 * D * D + D) * sizeof(float);
    if (cudaFuncSetAttribute(ahla_cross_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return -1;
    ahla_cross_kernel<TM><<<dim3(a.nseg - 1, a.BH), kScanThreads, smem, st>>>(a, a.seg_chunks * a.W);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

size_t ahla_chunk_smem(int d, int W) {
#define HLA2_AHLA_SMEM(DD, WW) \
    if (d == DD && W == WW) return AhlaCfg<DD, WW>::BYTES;
    HLA2_AHLA_SMEM(16, 32) HLA2_AHLA_SMEM(16, 64) HLA2_AHLA_SMEM(32, 32) HLA2_AHLA_SMEM(32, 64)
    HLA2_AHLA_SMEM(64, 32) HLA2_AHLA_SMEM(64, 64) HLA2_AHLA_SMEM(128, 32) HLA2_AHLA_SMEM(128, 64)
#undef HLA2_AHLA_SMEM
    return 0;
}

int ahla_chunk_threads(int d) { return 32 * (d <= 32 ? 4 : (d == 64 ? 8 : 16)); }

int launch_ahla_chunk(const AhlaArgs& a, int d, int W, bool summary, cudaStream_t st) {
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
#define HLA2_AHLA_CHUNK(DD, WW) \
    if (d == DD && W == WW) return launch_chunk_t<DD, WW>(a, summary, st);
    HLA2_AHLA_CHUNK(16, 32) HLA2_AHLA_CHUNK(16, 64) HLA2_AHLA_CHUNK(32, 32) HLA2_AHLA_CHUNK(32, 64)
    HLA2_AHLA_CHUNK(64, 32) HLA2_AHLA_CHUNK(64, 64) HLA2_AHLA_CHUNK(128, 32) HLA2_AHLA_CHUNK(128, 64)
#undef HLA2_AHLA_CHUNK
    return -2;
}

int launch_ahla_init(const AhlaArgs& a, int d, cudaStream_t st) {
    if (a.BH <= 0) return 0;
    ahla_init_kernel<<<a.BH, kScanThreads, 0, st>>>(a, d);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_ahla_cross(const AhlaArgs& a, int d, cudaStream_t st) {
    if (a.nseg <= 1 || a.BH <= 0) return 0;
    switch (d) {
        case 16: return launch_cross_t<1>(a, st);
        case 32: return launch_cross_t<2>(a, st);
        case 64: return launch_cross_t<4>(a, st);
        case 128: return launch_cross_t<8>(a, st);
        default: return -1;
    }
}

}  // namespace hla2
