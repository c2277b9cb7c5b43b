// bf16 reverse-mode chunk kernel of the masked HLA-2 backward (tensor cores,
// mma.m16n8k16).  Gradients of the unnormalised output, equal to those of the serial
// recurrence (page "Higher-order Linear Attention", section summary §4.2: a reverse-mode
// scan reproduces the serial recurrence's gradients).
//
// In the chained form p_t = S_t q_t, Z_t = g^2 Z_{t-1} + p_t v_t^T, o_t = q_t^T Z_t the
// adjoint is two reverse scans:
//     Zh_t = q_t dO_t^T + g^2 Zh_{t+1}          (d x dv)
//     dp_t = Zh_t v_t
//     Sh_t = dp_t q_t^T + g Sh_{t+1}            (d x d)
//     dq_t = Z_t dO_t + S_t dp_t,   dv_t = Zh_t^T p_t,   dk_t = (Sh_t + Sh_t^T) k_t.
// Per chunk (rows r = 0..Wc-1, forward state S0, Z0 at the chunk start, reverse carries
// Zh, Sh at the chunk end; Gam1[r,i] = [i <= r] g^(r-i), Gam2[r,j] = [j <= r] g^(2(r-j))):
//   A~ = (Q K^T) * Gam1,          P  = diag(g^(r+1)) Q S0 + A~ K
//   D~ = (dO V^T) * Gam2,         B~ = (Q P^T) * Gam2
//   dP = D~^T Q + diag(g^(2(Wc-1-j))) V Zh^T
//   dA~ = (dP K^T) * Gam1
//   dV = B~^T dO + diag(g^(2(Wc-1-j))) P Zh
//   dQ = D~ P + dA~ K + diag(g^(r+1)) (dP S0 + diag(g^(r+1)) dO Z0^T)
//   dK = A~^T dP + dA~^T Q + diag(g^(Wc-1-i)) K (Sh + Sh^T)
//   Zh <- g^(2Wc) Zh + Qh^T dO,   Qh = diag(g^(2(r+1))) Q
//   Sh <- g^Wc Sh + dPh^T Q,      dPh = diag(g^(r+1)) dP
// RSUM mode starts from zero carries and keeps only what the reverse scan needs
// (dP and the carry updates), storing the segment's reverse summary (Zh, Sh).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace hla2 {

template <int D, int DV, int W>
struct BwdCfg {
    static constexpr int NW = D <= 32 ? 4 : (D == 64 ? 8 : 16);
    static constexpr int NT = NW * 32;
    static constexpr int LD = D + 8, LDV = DV + 8, LW = W + 8;
    static constexpr int TW = W / 16, TD = D / 16, TV = DV / 16;
    static constexpr int S_TILES = TD * TD, Z_TILES = TD * TV;
    static constexpr int S_PER = (S_TILES + NW - 1) / NW;
    static constexpr int Z_PER = (Z_TILES + NW - 1) / NW;
    static constexpr size_t RD = (size_t)W * LD * 2, RV = (size_t)W * LDV * 2, RW = (size_t)W * LW * 2;
    static constexpr size_t oQ = 0, oK = oQ + RD, oV = oK + RD, oO = oV + RV, oQh = oO + RV;
    static constexpr size_t oAt = oQh + RD, oDt = oAt + RW, oBt = oDt + RW, odAt = oBt + RW;
    static constexpr size_t oP = odAt + RW, odP = oP + RD, odPh = odP + RD;
    static constexpr size_t oS0 = odPh + RD, oZ0 = oS0 + (size_t)D * LD * 2;
    static constexpr size_t oZh = oZ0 + (size_t)D * LDV * 2, oSh = oZh + (size_t)D * LDV * 2;
    static constexpr size_t oF = oSh + (size_t)D * LD * 2;
    static constexpr size_t BYTES = oF + ((size_t)(2 * W + 2) * 4 + 15) / 16 * 16;
};

template <int D, int DV, int W, bool RSUM>
__global__ void __launch_bounds__(BwdCfg<D, DV, W>::NT) bwd_chunk_mma_kernel(const BwdArgs a) {
    using Cfg = BwdCfg<D, DV, W>;
    constexpr int NW = Cfg::NW, NT = Cfg::NT, LD = Cfg::LD, LDV = Cfg::LDV, LW = Cfg::LW;
    constexpr int TW = Cfg::TW, TD = Cfg::TD, TV = Cfg::TV;
    extern __shared__ __align__(128) unsigned char smem[];
    bf16* Qs = reinterpret_cast<bf16*>(smem + Cfg::oQ);
    bf16* Ks = reinterpret_cast<bf16*>(smem + Cfg::oK);
    bf16* Vs = reinterpret_cast<bf16*>(smem + Cfg::oV);
    bf16* Os = reinterpret_cast<bf16*>(smem + Cfg::oO);  // dO
    bf16* Qh = reinterpret_cast<bf16*>(smem + Cfg::oQh);
    bf16* At = reinterpret_cast<bf16*>(smem + Cfg::oAt);
    bf16* Dt = reinterpret_cast<bf16*>(smem + Cfg::oDt);
    bf16* Bt = reinterpret_cast<bf16*>(smem + Cfg::oBt);
    bf16* dAt = reinterpret_cast<bf16*>(smem + Cfg::odAt);
    bf16* Ps = reinterpret_cast<bf16*>(smem + Cfg::oP);
    bf16* dPs = reinterpret_cast<bf16*>(smem + Cfg::odP);
    bf16* dPh = reinterpret_cast<bf16*>(smem + Cfg::odPh);
    bf16* S0s = reinterpret_cast<bf16*>(smem + Cfg::oS0);
    bf16* Z0s = reinterpret_cast<bf16*>(smem + Cfg::oZ0);
    bf16* Zhs = reinterpret_cast<bf16*>(smem + Cfg::oZh);
    bf16* Shs = reinterpret_cast<bf16*>(smem + Cfg::oSh);
    float* gp = reinterpret_cast<float*>(smem + Cfg::oF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int c_begin = seg * a.seg_chunks;
    const int c_end = min(c_begin + a.seg_chunks, a.nchunks);
    const size_t hq = (size_t)bh * a.n;
    const float log2g = log2f(head_decay(a.gamma, bh, a.H));
    for (int i = tid; i < 2 * W + 2; i += NT) gp[i] = pow_decay(log2g, (float)i);

    // reverse carries: fp32 tiles owned per warp
    float Zh[Cfg::Z_PER][2][4];
    float Sh[Cfg::S_PER][2][4];
    const size_t sidx = (size_t)bh * a.nseg + seg;
    const float* Zh0 = RSUM ? nullptr : a.ws + a.Zh_end + sidx * D * DV;
    const float* Sh0 = RSUM ? nullptr : a.ws + a.Sh_end + sidx * D * D;
#pragma unroll
    for (int s = 0; s < Cfg::Z_PER; ++s) {
        const int t = warp + s * NW;
        const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Zh[s][h][i] = (Zh0 && t < Cfg::Z_TILES) ? Zh0[(size_t)acc_row(m0, i) * DV + acc_col(n0, h, i)] : 0.f;
    }
#pragma unroll
    for (int s = 0; s < Cfg::S_PER; ++s) {
        const int t = warp + s * NW;
        const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Sh[s][h][i] = (Sh0 && t < Cfg::S_TILES) ? Sh0[(size_t)acc_row(m0, i) * D + acc_col(n0, h, i)] : 0.f;
    }

    auto publish_carries = [&]() {
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
            const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<uint32_t*>(&Zhs[acc_row(m0, i) * LDV + acc_col(n0, h, i)]) =
                        pack_bf16x2(Zh[s][h][i], Zh[s][h][i + 1]);
        }
        if (RSUM) return;
#pragma unroll
        for (int s = 0; s < Cfg::S_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::S_TILES) break;
            const int m0 = (t / TD) * 16, n0 = (t % TD) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<uint32_t*>(&Shs[acc_row(m0, i) * LD + acc_col(n0, h, i)]) =
                        pack_bf16x2(Sh[s][h][i], Sh[s][h][i + 1]);
        }
    };
    publish_carries();

    auto load_rows = [&](bf16* dst, int ld, const bf16* src, int width, int row0, int Wc) {
        const int cpr = width / 8;
        for (int i = tid; i < W * cpr; i += NT) {
            const int r = i / cpr, p = (i % cpr) * 8;
            if (r < Wc && HLA2_IN(row0 + r < a.n, 501))
                cp_async16(&dst[r * ld + p], src + (size_t)(row0 + r) * width + p);
            else
                *reinterpret_cast<uint4*>(&dst[r * ld + p]) = make_uint4(0, 0, 0, 0);
        }
    };
    auto load_chunk = [&](int c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        load_rows(Qs, LD, a.q + hq * D, D, row0, Wc);
        load_rows(Vs, LDV, a.v + hq * DV, DV, row0, Wc);
        load_rows(Os, LDV, a.dout + hq * DV, DV, row0, Wc);
        if (!RSUM && HLA2_IN(bh < a.BH && c < a.nchunks, 502)) {
            load_rows(Ks, LD, a.k + hq * D, D, row0, Wc);
            const bf16* st = a.chunk_states + ((size_t)bh * a.nchunks + c) * (size_t)(D * D + D * DV);
            for (int i = tid; i < D * D / 8; i += NT) {
                const int r = (i * 8) / D, f = (i * 8) % D;
                cp_async16(&S0s[r * LD + f], st + (size_t)r * D + f);
            }
            for (int i = tid; i < D * DV / 8; i += NT) {
                const int r = (i * 8) / DV, f = (i * 8) % DV;
                cp_async16(&Z0s[r * LDV + f], st + (size_t)D * D + (size_t)r * DV + f);
            }
        }
        cp_async_commit();
    };
    if (c_begin < c_end) load_chunk(c_end - 1);

    for (int c = c_end - 1; c >= c_begin; --c) {
        const int row0 = c * W, Wc = min(W, a.n - row0);
        cp_async_wait_all();
        __syncthreads();

        // ---- phase 1: Qh; A~ = mask(Q K^T); D~ = mask2(dO V^T) ---------------------
        for (int i = tid; i < W * D; i += NT) {
            const int r = i / D, f = i % D;
            Qh[r * LD + f] = from_f32<bf16>((r < Wc ? gp[2 * (r + 1)] : 0.f) * to_f32(Qs[r * LD + f]));
        }
        for (int t = warp; t < 2 * TW * TW; t += NW) {
            const bool isD = t >= TW * TW;
            if (RSUM && !isD) continue;
            const int tt = isD ? t - TW * TW : t;
            const int rb = tt / TW, cb = tt % TW;
            if (cb > rb) continue;
            float acc[2][4];
            zero_acc(acc);
            if (isD)
                warp_tile_mma<false, false>(acc, Os, LDV, rb * 16, Vs, LDV, cb * 16, 0, DV);
            else
                warp_tile_mma<false, false>(acc, Qs, LD, rb * 16, Ks, LD, cb * 16, 0, D);
            bf16* dst = isD ? Dt : At;
            const int p2 = isD ? 2 : 1;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2) {
                    const int r = acc_row(rb * 16, i), col = acc_col(cb * 16, h, i);
                    const float v0 = col <= r ? gp[p2 * (r - col)] * acc[h][i] : 0.f;
                    const float v1 = col + 1 <= r ? gp[p2 * (r - col - 1)] * acc[h][i + 1] : 0.f;
                    *reinterpret_cast<uint32_t*>(&dst[r * LW + col]) = pack_bf16x2(v0, v1);
                }
        }
        __syncthreads();

        // ---- phase 2: P (forward recompute), dP, dPh -----------------------------------
        for (int t = warp; t < 2 * TW * TD; t += NW) {
            const bool isdP = t >= TW * TD;
            if (RSUM && !isdP) continue;
            const int tt = isdP ? t - TW * TD : t;
            const int rb = tt / TD, fb = tt % TD;
            float acc[2][4];
            zero_acc(acc);
            if (!isdP) {
                warp_tile_mma<false, true>(acc, Qs, LD, rb * 16, S0s, LD, fb * 16, 0, D);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
                warp_tile_mma<false, true>(acc, At, LW, rb * 16, Ks, LD, fb * 16, 0, (rb + 1) * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(fb * 16, h, i);
                        *reinterpret_cast<uint32_t*>(&Ps[r * LD + col]) = pack_bf16x2(acc[h][i], acc[h][i + 1]);
                    }
            } else {
                // rows j: g^(2(Wc-1-j)) (V Zh^T)[j] + sum_{r >= j} D~[r, j] q_r
                warp_tile_mma<false, false>(acc, Vs, LDV, rb * 16, Zhs, LDV, fb * 16, 0, DV);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int j = acc_row(rb * 16, i);
                        acc[h][i] *= j < Wc ? gp[2 * (Wc - 1 - j)] : 0.f;
                    }
                warp_tile_mma<true, true>(acc, Dt, LW, rb * 16, Qs, LD, fb * 16, rb * 16, W);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int j = acc_row(rb * 16, i), col = acc_col(fb * 16, h, i);
                        const float w1 = j < Wc ? gp[j + 1] : 0.f;
                        *reinterpret_cast<uint32_t*>(&dPs[j * LD + col]) = pack_bf16x2(acc[h][i], acc[h][i + 1]);
                        *reinterpret_cast<uint32_t*>(&dPh[j * LD + col]) =
                            pack_bf16x2(w1 * acc[h][i], w1 * acc[h][i + 1]);
                    }
            }
        }
        __syncthreads();

        if (!RSUM) {
            // ---- phase 3: B~ = mask2(Q P^T); dA~ = mask1(dP K^T) ---------------------------
            for (int t = warp; t < 2 * TW * TW; t += NW) {
                const bool isdA = t >= TW * TW;
                const int tt = isdA ? t - TW * TW : t;
                const int rb = tt / TW, cb = tt % TW;
                if (cb > rb) continue;
                float acc[2][4];
                zero_acc(acc);
                if (isdA)
                    warp_tile_mma<false, false>(acc, dPs, LD, rb * 16, Ks, LD, cb * 16, 0, D);
                else
                    warp_tile_mma<false, false>(acc, Qs, LD, rb * 16, Ps, LD, cb * 16, 0, D);
                bf16* dst = isdA ? dAt : Bt;
                const int p2 = isdA ? 1 : 2;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(cb * 16, h, i);
                        const float v0 = col <= r ? gp[p2 * (r - col)] * acc[h][i] : 0.f;
                        const float v1 = col + 1 <= r ? gp[p2 * (r - col - 1)] * acc[h][i + 1] : 0.f;
                        *reinterpret_cast<uint32_t*>(&dst[r * LW + col]) = pack_bf16x2(v0, v1);
                    }
            }
            __syncthreads();

            // ---- phase 4: dV, dQ, dK -> global ------------------------------------------------
            constexpr int NV = TW * TV, NQ = TW * TD;
            for (int t = warp; t < NV + 2 * NQ; t += NW) {
                float acc[2][4];
                zero_acc(acc);
                bf16* dst;
                int ldo, rb, cb;
                if (t < NV) {  // dV rows j
                    rb = t / TV;
                    cb = t % TV;
                    warp_tile_mma<false, true>(acc, Ps, LD, rb * 16, Zhs, LDV, cb * 16, 0, D);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int j = acc_row(rb * 16, i);
                            acc[h][i] *= j < Wc ? gp[2 * (Wc - 1 - j)] : 0.f;
                        }
                    warp_tile_mma<true, true>(acc, Bt, LW, rb * 16, Os, LDV, cb * 16, rb * 16, W);
                    dst = a.dv + (hq + row0) * DV;
                    ldo = DV;
                } else if (t < NV + NQ) {  // dQ rows r
                    const int tt = t - NV;
                    rb = tt / TD;
                    cb = tt % TD;
                    warp_tile_mma<false, false>(acc, Os, LDV, rb * 16, Z0s, LDV, cb * 16, 0, DV);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
                    warp_tile_mma<false, true>(acc, dPs, LD, rb * 16, S0s, LD, cb * 16, 0, D);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[h][i] *= gp[acc_row(rb * 16, i) + 1];
                    warp_tile_mma<false, true>(acc, Dt, LW, rb * 16, Ps, LD, cb * 16, 0, (rb + 1) * 16);
                    warp_tile_mma<false, true>(acc, dAt, LW, rb * 16, Ks, LD, cb * 16, 0, (rb + 1) * 16);
                    dst = a.dq + (hq + row0) * D;
                    ldo = D;
                } else {  // dK rows i
                    const int tt = t - NV - NQ;
                    rb = tt / TD;
                    cb = tt % TD;
                    warp_tile_mma<false, true>(acc, Ks, LD, rb * 16, Shs, LD, cb * 16, 0, D);
                    warp_tile_mma<false, false>(acc, Ks, LD, rb * 16, Shs, LD, cb * 16, 0, D);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int ii = acc_row(rb * 16, i);
                            acc[h][i] *= ii < Wc ? gp[Wc - 1 - ii] : 0.f;
                        }
                    warp_tile_mma<true, true>(acc, At, LW, rb * 16, dPs, LD, cb * 16, rb * 16, W);
                    warp_tile_mma<true, true>(acc, dAt, LW, rb * 16, Qs, LD, cb * 16, rb * 16, W);
                    dst = a.dk + (hq + row0) * D;
                    ldo = D;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; i += 2) {
                        const int r = acc_row(rb * 16, i), col = acc_col(cb * 16, h, i);
                        if (r < Wc && HLA2_IN(row0 + r < a.n, 503))
                            *reinterpret_cast<uint32_t*>(&dst[(size_t)r * ldo + col]) = pack_bf16x2(acc[h][i], acc[h][i + 1]);
                    }
            }
        }

        // ---- carries to the chunk start (registers) -----------------------------------------
        const float rho = gp[Wc], rho2 = gp[2 * Wc];
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) Zh[s][h][i] *= rho2;
            warp_tile_mma<true, true>(Zh[s], Qh, LD, (t / TV) * 16, Os, LDV, (t % TV) * 16, 0, W);
        }
#pragma unroll
        for (int s = 0; s < Cfg::S_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::S_TILES) break;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) Sh[s][h][i] *= rho;
            warp_tile_mma<true, true>(Sh[s], dPh, LD, (t / TD) * 16, Qs, LD, (t % TD) * 16, 0, W);
        }
        __syncthreads();
        publish_carries();
        if (c > c_begin) load_chunk(c - 1);
    }

    if (RSUM && HLA2_IN(bh < a.BH && seg < a.nseg, 504)) {
        float* dZ = a.ws + a.ZhB + sidx * D * DV;
        float* dS = a.ws + a.ShB + sidx * D * D;
#pragma unroll
        for (int s = 0; s < Cfg::Z_PER; ++s) {
            const int t = warp + s * NW;
            if (t >= Cfg::Z_TILES) break;
            const int m0 = (t / TV) * 16, n0 = (t % TV) * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; i += 2)
                    *reinterpret_cast<float2*>(&dZ[(size_t)acc_row(m0, i) * DV + acc_col(n0, h, i)]) =
                        make_float2(Zh[s][h][i], Zh[s][h][i + 1]);
        }
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
                        make_float2(Sh[s][h][i], Sh[s][h][i + 1]);
        }
    }
    (void)lane;
}

template <int D, int DV, int W>
int launch_bwd_chunk_mma_t(const BwdArgs& a, bool rsum, cudaStream_t st) {
    using Cfg = BwdCfg<D, DV, W>;
    if (a.nseg <= 0 || a.BH <= 0) return 0;
    const size_t smem = Cfg::BYTES;
    auto kfn = rsum ? bwd_chunk_mma_kernel<D, DV, W, true> : bwd_chunk_mma_kernel<D, DV, W, false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -1;
    kfn<<<dim3(a.nseg, a.BH), Cfg::NT, smem, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace hla2
