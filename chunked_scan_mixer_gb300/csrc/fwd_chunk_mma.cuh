// bf16 chunk kernel of the masked HLA-2 forward (tensor cores, mma.m16n8k16).
//
// One CTA walks the chunks of one segment of one head in time order, keeping the
// segment's running state in fp32 registers.  It works in the "two chained scans"
// form of the masked output:
//     p_t = S_t q_t                       (S_t = g S_{t-1} + k_t k_t^T)
//     Z_t = g^2 Z_{t-1} + p_t v_t^T,      o_t = q_t^T Z_t
//     y_t = g^2 y_{t-1} + p_t,            den_t = q_t^T y_t
// which equals the paper's o_t = q_t^T (S_t C_t - G_t) with Z_t = S_t C_t - G_t and
// y_t = S_t m_t - h_t (page "Higher-order Linear Attention", technical summary item
// "1. Zweite Ordnung HLA"; the identity is checked against the float64 oracle).
//
// Per chunk of width W (local rows r = 0..Wc-1, state at the chunk start S0, Z0, y0):
//   A~ = (Q K^T) * [i <= r] g^(r-i)                    masked dense chunk product
//   P  = diag(g^(r+1)) Q S0 + A~ K                     p for every token
//   B~ = (Q P^T) * [j <= r] g^(2(r-j))
//   O  = diag(g^(2(r+1))) Q Z0 + B~ V;  den = diag(g^(2(r+1))) Q y0 + B~ 1
//   S  <- g^Wc S0 + K~^T K,    K~ = diag(g^(Wc-1-i)) K
//   Z  <- g^(2Wc) Z0 + P~^T V, P~ = diag(g^(2(Wc-1-j))) P;   y likewise with V -> 1
//   C  <- g^Wc C0 + Q~^T V,    Q~ = diag(g^(Wc-1-j)) Q;      m likewise
// kSummary starts from zero and stores (S, C, Z, m, y) of the segment (its summary
// for the inter-segment scan); kOutput starts from the segment's carry-in and writes
// out (and the raw final state for the last segment); kStates starts from the carry-in
// and exports the bf16 (S, Z) at every chunk start (the forward states that the
// reverse-mode pass consumes); kOutStates does both (the forward of a training step).
//
// UM selects the unmasked output o_t = q_t^T S_t C_t = p_t^T C_t (section summary §3,
// the bilinear form without the G correction; its scan is the unmasked monoid of §4.1).
// It is a first-order scan with queries p, keys q and values v, so per chunk
//   B~ = (P Q^T) * [j <= r] g^(r-j),   O = diag(g^(r+1)) P C0 + B~ V,
//   den = diag(g^(r+1)) P m0 + B~ 1,   C <- g^Wc C0 + Q~^T V,   m likewise,
// and the Z and y registers, tiles and workspace slots hold C and m instead.  The
// summary pass then needs no A~ and no P at all.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace hla2 {

template <int D, int DV, int W>
struct MmaCfg {
    static constexpr int NW = D <= 32 ? 4 : (D == 64 ? 8 : 16);
    static constexpr int NT = NW * 32;
    static constexpr int LD = D + 8;    // bf16 row strides (16-byte pad)
    static constexpr int LDV = DV + 8;
    static constexpr int LW = W + 8;
    static constexpr int TW = W / 16, TD = D / 16, TV = DV / 16;
    static constexpr int S_TILES = TD * TD, Z_TILES = TD * TV;
    static constexpr int S_PER = (S_TILES + NW - 1) / NW;
    static constexpr int Z_PER = (Z_TILES + NW - 1) / NW;
    // shared memory carve-up (bytes)
    static constexpr size_t ROWS_D = (size_t)W * LD * 2, ROWS_V = (size_t)W * LDV * 2;
    static constexpr size_t oQ = 0, oK = oQ + ROWS_D, oV = oK + ROWS_D, oKt = oV + ROWS_V;
    static constexpr size_t oP = oKt + ROWS_D, oPt = oP + ROWS_D;
    static constexpr size_t oAB = oPt + ROWS_D;
    static constexpr size_t oS = oAB + (size_t)W * LW * 2;
    static constexpr size_t oZ = oS + (size_t)D * LD * 2;
    static constexpr size_t oF = oZ + (size_t)D * LDV * 2;  // float region
    // floats: gp[2W+2] den[W] denpart[TW][W] ypart[TW][D] y[D] m[D]; the per-tile partial
    // sums of the denominator rows and the y increment are added in a fixed order, so that
    // the result does not depend on the order in which warps finish
    static constexpr size_t nF = (2 * W + 2) + W + (size_t)TW * W + (size_t)TW * D + 2 * D;
    static constexpr size_t oQt = oF + ((nF * 4 + 15) / 16) * 16;
    static constexpr size_t bytes(bool cm) { return oQt + (cm ? ROWS_D : 0); }
};

template <int D, int DV, int W, int MODE, bool CM, bool UM>
__global__ void __launch_bounds__(MmaCfg<D, DV, W>::NT)
    fwd_chunk_mma_kernel(const ChunkArgs a) {
    static_assert(!UM || (!CM && (MODE == kSummary || MODE == kOutput)), "unmasked: summary and output passes only");
    constexpr bool SUMMARY = MODE == kSummary, OUTPUT = MODE == kOutput || MODE == kOutStates;
    constexpr bool NEED_P = !(UM && SUMMARY);  // the unmasked summary needs no p
    constexpr bool EXPORT = MODE == kStates || MODE == kOutStates;
    using Cfg = MmaCfg<D, DV, W>;
    constexpr int NW = Cfg::NW, NT = Cfg::NT, LD = Cfg::LD, LDV = Cfg::LDV, LW = Cfg::LW;
    constexpr int TW = Cfg::TW, TD = Cfg::TD, TV = Cfg::TV;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16* Qs = reinterpret_cast<bf16*>(smem + Cfg::oQ);
    bf16* Ks = reinterpret_cast<bf16*>(smem + Cfg::oK);
    bf16* Vs = reinterpret_cast<bf16*>(smem + Cfg::oV);
    bf16* Kt = reinterpret_cast<bf16*>(smem + Cfg::oKt);
    bf16* Ps = reinterpret_cast<bf16*>(smem + Cfg::oP);
    bf16* Pt = reinterpret_cast<bf16*>(smem + Cfg::oPt);
    bf16* AB = reinterpret_cast<bf16*>(smem + Cfg::oAB);
    bf16* Sst = reinterpret_cast<bf16*>(smem + Cfg::oS);
    bf16* Zst = reinterpret_cast<bf16*>(smem + Cfg::oZ);
    float* gp = reinterpret_cast<float*>(smem + Cfg::oF);
    float* den = gp + 2 * W + 2;
    float* denpart = den + W;          // [TW][W]: row sums of B~ over column block jb
    float* ypart = denpart + TW * W;   // [TW][D]: column sums of P~ over row block rb
    float* ys = ypart + TW * D;
    float* ms = ys + D;
    bf16* Qt = reinterpret_cast<bf16*>(smem + Cfg::oQt);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = a.seg0 + blockIdx.x, bh = blockIdx.y;
    const int nseg = a.nseg;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const bool last_seg = (seg == nseg - 1);
    const bf16* q = static_cast<const bf16*>(a.q) + (size_t)bh * a.n * D;
    const bf16* k = static_cast<const bf16*>(a.k) + (size_t)bh * a.n * D;
    const bf16* v = static_cast<const bf16*>(a.v) + (size_t)bh * a.n * DV;

    const float g = head_decay(a.gamma, bh, a.H);
    const float log2g = log2f(g);
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);

    // ---- running state: fp32 accumulators owned per warp -------------------------
    float Sacc[Cfg::S_PER][2][4];
    float Zacc[Cfg::Z_PER][2][4];
    float Cacc[CM ? Cfg::Z_PER : 1][2][4];
    const float* Sinit = nullptr;
    const float* Zinit = nullptr;
    const float* Cinit = nullptr;
    if (!SUMMARY) {
        const size_t sidx = (size_t)bh * nseg + seg;
        if (HLA2_IN(a.L.Sin + (sidx + 1) * D * D <= a.L.total && a.L.Zin + (sidx + 1) * D * DV <= a.L.total &&
                        a.L.Clast + (size_t)(bh + 1) * D * DV <= a.L.total,
                    401)) {
            Sinit = a.ws + a.L.Sin + sidx * D * D;
            Zinit = a.ws + a.L.Zin + sidx * D * DV;
            if (CM) Cinit = a.ws + a.L.Clast + (size_t)bh * D * DV;
        }
    }
#pragma unroll
    for (int s = 0; s < Cfg::S_PER; ++s) {
        const int t = warp + s * NW;
        const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Sacc[s][h][i] = (Sinit && t < Cfg::S_TILES)
                                    ? Sinit[(size_t)acc_row(m0, i) * D + acc_col(n0, h, i)]
                                    : 0.f;
    }
#pragma unroll
    for (int s = 0; s < Cfg::Z_PER; ++s) {
        const int t = warp + s * NW;
        const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const size_t e = (size_t)acc_row(m0, i) * DV + acc_col(n0, h, i);
                const bool ok = t < Cfg::Z_TILES;
                Zacc[s][h][i] = (Zinit && ok) ? Zinit[e] : 0.f;
                if (CM) Cacc[s][h][i] = (Cinit && ok) ? Cinit[e] : 0.f;
            }
    }
    for (int f = tid; f < D; f += NT) {
        ys[f] = SUMMARY ? 0.f : a.ws[a.L.yin + ((size_t)bh * nseg + seg) * D + f];
        ms[f] = (CM && !SUMMARY) ? a.ws[a.L.mlast + (size_t)bh * D + f] : 0.f;
    }
    for (int i = tid; i < TW * D; i += NT) ypart[i] = 0.f;

    // bf16 copies of S and Z: the B operands of Q S0 and Q Z0
    auto publish_state = [&]() {
#pragma unroll
        for (int s = 0; s < Cfg::S_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::S_TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<uint32_t*>(&Sst[acc_row(m0, i) * LD + acc_col(n0, h, i)]) =
                        pack_bf16x2(Sacc[s][h][i], Sacc[s][h][i + 1]);
        }
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
            const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<uint32_t*>(&Zst[acc_row(m0, i) * LDV + acc_col(n0, h, i)]) =
                        pack_bf16x2(Zacc[s][h][i], Zacc[s][h][i + 1]);
        }
    };
    publish_state();

    // chunk loads: rows < Wc by cp.async, rows >= Wc zero-filled
    auto load_chunk = [&](int c) {
        const int row0 = c * W;
        const int Wc = min(W, a.n - row0);
        constexpr int CPR = D / 8, CPRV = DV / 8;  // 16-byte pieces per row
        for (int i = tid; i < W * CPR; i += NT) {
            const int r = i / CPR, p = (i % CPR) * 8;
            if (r < Wc && HLA2_IN(row0 + r < a.n, 402)) {
                cp_async16(&Qs[r * LD + p], q + (size_t)(row0 + r) * D + p);
                cp_async16(&Ks[r * LD + p], k + (size_t)(row0 + r) * D + p);
            } else {
                *reinterpret_cast<uint4*>(&Qs[r * LD + p]) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(&Ks[r * LD + p]) = make_uint4(0, 0, 0, 0);
            }
        }
        for (int i = tid; i < W * CPRV; i += NT) {
            const int r = i / CPRV, p = (i % CPRV) * 8;
            if (r < Wc && HLA2_IN(row0 + r < a.n, 403))
                cp_async16(&Vs[r * LDV + p], v + (size_t)(row0 + r) * DV + p);
            else
                *reinterpret_cast<uint4*>(&Vs[r * LDV + p]) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
    };
    if (c_begin < c_end) load_chunk(c_begin);

    for (int c = c_begin; c < c_end; ++c) {
        const int Wc = min(W, a.n - c * W);
        cp_async_wait_all();
        __syncthreads();

        if (EXPORT && HLA2_IN(bh < a.BH && c < a.nchunks, 404)) {  // export the state at this chunk start
            bf16* dst = a.chunk_states + ((size_t)bh * a.nchunks + c) * (size_t)(D * D + D * DV);
            for (int i = tid; i < D * D / 8; i += NT) {
                const int r = (i * 8) / D, f = (i * 8) % D;
                *reinterpret_cast<uint4*>(dst + (size_t)r * D + f) = *reinterpret_cast<const uint4*>(&Sst[r * LD + f]);
            }
            for (int i = tid; i < D * DV / 8; i += NT) {
                const int r = (i * 8) / DV, f = (i * 8) % DV;
                *reinterpret_cast<uint4*>(dst + (size_t)D * D + (size_t)r * DV + f) =
                    *reinterpret_cast<const uint4*>(&Zst[r * LDV + f]);
            }
        }

        // ---- scaled copies, query mass, denominator carry term ----------------------
        for (int i = tid; i < W * D; i += NT) {
            const int r = i / D, f = i % D;
            const float w1 = r < Wc ? gp[Wc - 1 - r] : 0.f;
            Kt[r * LD + f] = from_f32<bf16>(w1 * to_f32(Ks[r * LD + f]));
            if (CM) Qt[r * LD + f] = from_f32<bf16>(w1 * to_f32(Qs[r * LD + f]));
            if (UM) Pt[r * LD + f] = from_f32<bf16>(w1 * to_f32(Qs[r * LD + f]));  // Q~
        }
        if (UM) {  // the query-mass increment, added to m (held in ys) after the chunk
            for (int f = tid; f < D; f += NT) {
                float s = 0.f;
                for (int r = 0; r < Wc; ++r) s += gp[Wc - 1 - r] * to_f32(Qs[r * LD + f]);
                ypart[f] = s;
            }
        }
        if (OUTPUT && a.normalize && !UM) {
            for (int r = tid; r < W; r += NT) {
                float s = 0.f;
                for (int f = 0; f < D; ++f) s += to_f32(Qs[r * LD + f]) * ys[f];
                den[r] = gp[2 * (r + 1)] * s;
            }
        }
        if (CM) {
            for (int f = tid; f < D; f += NT) {
                float s = 0.f;
                for (int r = 0; r < Wc; ++r) s += gp[Wc - 1 - r] * to_f32(Qs[r * LD + f]);
                ms[f] = gp[Wc] * ms[f] + s;
            }
        }
        __syncthreads();

        // ---- A~ = mask(Q K^T) ---------------------------------------------------------
        for (int t = warp; NEED_P && t < TW * TW; t += NW) {
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

        // ---- P = diag(g^(r+1)) Q S0 + A~ K ; P~ ; y increment -------------------------
        for (int t = warp; NEED_P && t < TW * TD; t += NW) {
            const int rb = t / TD, fb = t % TD;
            float acc[2][4];
            zero_acc(acc);
            warp_tile_mma<false, true>(acc, Qs, LD, rb * 16, Sst, LD, fb * 16, 0, D);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
            warp_tile_mma<false, true>(acc, AB, LW, rb * 16, Ks, LD, fb * 16, 0, (rb + 1) * 16);
            float colsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int r = acc_row(rb * 16, i), col = acc_col(fb * 16, h, i);
                    *reinterpret_cast<uint32_t*>(&Ps[r * LD + col]) = pack_bf16x2(acc[h][i], acc[h][i + 1]);
                    if (UM) continue;
                    const float w2 = r < Wc ? gp[2 * (Wc - 1 - r)] : 0.f;
                    *reinterpret_cast<uint32_t*>(&Pt[r * LD + col]) =
                        pack_bf16x2(w2 * acc[h][i], w2 * acc[h][i + 1]);
                    colsum[h][0] += w2 * acc[h][i];
                    colsum[h][1] += w2 * acc[h][i + 1];
                }
            if (UM) continue;
            // reduce the 16 rows of the tile: lanes with equal (lane & 3) share columns
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float s = colsum[h][j];
                    s += __shfl_xor_sync(0xffffffffu, s, 4);
                    s += __shfl_xor_sync(0xffffffffu, s, 8);
                    s += __shfl_xor_sync(0xffffffffu, s, 16);
                    if (lane < 4) ypart[rb * D + fb * 16 + h * 8 + lane * 2 + j] = s;
                }
        }
        __syncthreads();

        if (OUTPUT && UM && a.normalize) {  // denominator carry term g^(r+1) p_r . m0
            for (int r = tid; r < W; r += NT) {
                float s = 0.f;
                for (int f = 0; f < D; ++f) s += to_f32(Ps[r * LD + f]) * ys[f];
                den[r] = gp[r + 1] * s;
            }
            __syncthreads();
        }

        if (OUTPUT) {
            // ---- B~ = mask(Q P^T) (+ row sums for the denominator); unmasked mask(P Q^T) --
            constexpr int BP = UM ? 1 : 2;  // decay power of the second scan
            for (int t = warp; t < TW * TW; t += NW) {
                const int rb = t / TW, jb = t % TW;
                if (jb > rb) continue;
                float acc[2][4];
                zero_acc(acc);
                if (UM)
                    warp_tile_mma<false, false>(acc, Ps, LD, rb * 16, Qs, LD, jb * 16, 0, D);
                else
                    warp_tile_mma<false, false>(acc, Qs, LD, rb * 16, Ps, LD, jb * 16, 0, D);
                float rs[2] = {0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(jb * 16, h, i);
                        const float v0 = col <= r ? gp[BP * (r - col)] * acc[h][i] : 0.f;
                        const float v1 = col + 1 <= r ? gp[BP * (r - col - 1)] * acc[h][i + 1] : 0.f;
                        *reinterpret_cast<uint32_t*>(&AB[r * LW + col]) = pack_bf16x2(v0, v1);
                        rs[i >> 1] += v0 + v1;
                    }
                if (a.normalize) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float s = rs[j];
                        s += __shfl_xor_sync(0xffffffffu, s, 1);
                        s += __shfl_xor_sync(0xffffffffu, s, 2);
                        if ((lane & 3) == 0) denpart[jb * W + rb * 16 + (lane >> 2) + j * 8] = s;
                    }
                }
            }
            __syncthreads();

            // ---- O = diag(g^(2(r+1))) Q Z0 + B~ V -> out; unmasked g^(r+1) P C0 + B~ V --
            bf16* outp = static_cast<bf16*>(a.out) + ((size_t)bh * a.n + (size_t)c * W) * DV;
            for (int t = warp; t < TW * TV; t += NW) {
                const int rb = t / TV, eb = t % TV;
                float acc[2][4];
                zero_acc(acc);
                warp_tile_mma<false, true>(acc, UM ? Ps : Qs, LD, rb * 16, Zst, LDV, eb * 16, 0, D);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[h][i] *= gp[BP * (acc_row(rb * 16, i) + 1)];
                warp_tile_mma<false, true>(acc, AB, LW, rb * 16, Vs, LDV, eb * 16, 0, (rb + 1) * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(eb * 16, h, i);
                        if (r >= Wc || !HLA2_IN(c * W + r < a.n, 405)) continue;
                        float o0 = acc[h][i], o1 = acc[h][i + 1];
                        if (a.normalize) {
                            float dr = den[r];
                            for (int jb = 0; jb <= r / 16; ++jb) dr += denpart[jb * W + r];
                            const float inv = 1.f / (dr + a.eps);
                            o0 *= inv;
                            o1 *= inv;
                        }
                        *reinterpret_cast<uint32_t*>(&outp[(size_t)r * DV + col]) = pack_bf16x2(o0, o1);
                    }
            }
        }

        // ---- state updates in registers (unmasked: Zacc holds C, Pt holds Q~) ---------------
        const float rho = gp[Wc], rho2 = gp[UM ? Wc : 2 * Wc];
#pragma unroll
        for (int s = 0; s < Cfg::S_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::S_TILES) break;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) Sacc[s][h][i] *= rho;
            warp_tile_mma<true, true>(Sacc[s], Kt, LD, (t / TD) * 16, Ks, LD, (t % TD) * 16, 0, W);
        }
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
            const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) Zacc[s][h][i] *= rho2;
            warp_tile_mma<true, true>(Zacc[s], Pt, LD, m0, Vs, LDV, n0, 0, W);
            if (CM) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) Cacc[s][h][i] *= rho;
                warp_tile_mma<true, true>(Cacc[s], Qt, LD, m0, Vs, LDV, n0, 0, W);
            }
        }
        __syncthreads();  // every read of Sst, Zst and the chunk tiles is done

        publish_state();
        for (int f = tid; f < D; f += NT) {
            float inc = 0.f;
            for (int rb = 0; rb < TW; ++rb) {
                inc += ypart[rb * D + f];
                ypart[rb * D + f] = 0.f;
            }
            ys[f] = rho2 * ys[f] + inc;
        }
        if (c + 1 < c_end) load_chunk(c + 1);
    }
    __syncthreads();

    // ---- epilogue: segment summary, or the raw final state --------------------------------
    float *dS = nullptr, *dC = nullptr, *dZ = nullptr, *dm = nullptr, *dy = nullptr;
    if (SUMMARY) {
        const size_t sidx = (size_t)bh * a.nsum + seg;
        dS = a.ws + a.L.SB + sidx * D * D;
        dC = a.ws + a.L.CB + sidx * D * DV;
        dZ = a.ws + a.L.ZB + sidx * D * DV;
        dm = a.ws + a.L.mB + sidx * D;
        dy = a.ws + a.L.yB + sidx * D;
    } else if (OUTPUT && (CM || UM) && last_seg && a.want_final) {
        const RawOff ro = raw_off(D, DV);
        float* base = a.ws + a.L.fin + (size_t)bh * raw_state_floats(D, DV);
        dS = base + ro.S;
        dC = base + ro.C;
        dZ = base + ro.Z;
        dm = base + ro.m;
        dy = base + ro.y;
    }
    if (dS && HLA2_IN(dS >= a.ws && (size_t)(dy + D - a.ws) <= a.L.total, 406)) {
#pragma unroll
        for (int s = 0; s < Cfg::S_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::S_TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<float2*>(&dS[(size_t)acc_row(m0, i) * D + acc_col(n0, h, i)]) =
                        make_float2(Sacc[s][h][i], Sacc[s][h][i + 1]);
        }
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
            const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const size_t e = (size_t)acc_row(m0, i) * DV + acc_col(n0, h, i);
                    *reinterpret_cast<float2*>(&dZ[e]) = make_float2(Zacc[s][h][i], Zacc[s][h][i + 1]);
                    if (CM) *reinterpret_cast<float2*>(&dC[e]) = make_float2(Cacc[s][h][i], Cacc[s][h][i + 1]);
                }
        }
        for (int f = tid; f < D; f += NT) {
            dm[f] = ms[f];
            dy[f] = ys[f];
        }
    }
}

template <int D, int DV, int W, int MODE, bool CM, bool UM = false>
cudaError_t launch_mode(const ChunkArgs& a, size_t smem, cudaStream_t st) {
    auto kfn = fwd_chunk_mma_kernel<D, DV, W, MODE, CM, UM>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kfn<<<dim3(a.nseg_launch, a.BH), MmaCfg<D, DV, W>::NT, smem, st>>>(a);
    return cudaPeekAtLastError();
}

template <int D, int DV, int W>
int launch_fwd_chunk_mma_t(const ChunkArgs& a, int mode, bool track_cm, cudaStream_t st) {
    using Cfg = MmaCfg<D, DV, W>;
    const bool cm = !a.unmasked && (mode == kSummary || track_cm);
    const size_t smem = Cfg::bytes(cm);
    if (a.nseg_launch <= 0 || a.BH <= 0) return 0;
    cudaError_t e;
    if (a.unmasked) {
        if (mode == kSummary)
            e = launch_mode<D, DV, W, kSummary, false, true>(a, smem, st);
        else if (mode == kOutput)
            e = launch_mode<D, DV, W, kOutput, false, true>(a, smem, st);
        else
            return -2;
    } else if (mode == kSummary)
        e = launch_mode<D, DV, W, kSummary, true>(a, smem, st);
    else if (mode == kStates)
        e = launch_mode<D, DV, W, kStates, false>(a, smem, st);
    else if (mode == kOutStates)
        e = launch_mode<D, DV, W, kOutStates, false>(a, smem, st);
    else if (track_cm)
        e = launch_mode<D, DV, W, kOutput, true>(a, smem, st);
    else
        e = launch_mode<D, DV, W, kOutput, false>(a, smem, st);
    return e == cudaSuccess ? 0 : -1;
}

template <int D, int DV, int W>
size_t fwd_chunk_mma_smem_t(bool track_cm) {
    return MmaCfg<D, DV, W>::bytes(track_cm);
}

}  // namespace hla2
