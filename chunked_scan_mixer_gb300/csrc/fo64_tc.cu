// First-order chunked linear attention on the 5th-generation tensor cores, d = dv = 64, chunk
// width 128 (bf16 tiles, fp32 state): the same passes as fo_tc.cu (d = dv = 128), with the
// tiles small enough (16 KB) that one CTA per SM keeps every input two chunks ahead.
//
// Per chunk of W = 128 rows r (Wc valid), with decay g (gamma or gamma^2 of the head):
//   MMA-G  G = X K^T                                        (128 x 128 fp32, tensor memory)
//   EPI-1  G~ = mask(G) (forward [i <= r] g^(r-i), reverse [i >= r] g^(i-r)), bf16 packed beside
//          fX = diag(f_r) X (forward f = g^(r+1), reverse g^(Wc-r));  K~ = diag(w_i) K (shared
//          memory; forward w = g^(Wc-1-i), reverse g^i)
//   MMA-Y  Y = [G~ | fX] [V ; Sig0]                         (N = 64, one accumulation)
//   MMA-S  dSig = [K~^T ; K~^T] V: the 64 x 64 increment as an M = 128 product whose two row
//          halves read the same K~ (so every epilogue thread owns 16 of its entries)
//   EPI-S  Sig <- g^Wc Sig + dSig (fp32, 16 a thread), bf16 Sig0 for the next chunk
//   EPI-Y  Y (+ a partial read from global) -> bf16 tile -> one TMA tile store
// Optional parts as in fo_tc.cu: the swapped second pair (R2), the next summary over the
// output (NSUM; the values are the value tile or an extra tile), a partial output (ADD).  Here
// also a second query / key pair with the same values (ST): out = (R)LA(X, K, V) + (R)LA(X2, K2, V)
// is one scan of the stacked pairs, G = X K^T + X2 K2^T, Y = [G~ | fX | fX2] [V ; Sig0 ; Sig0_2],
// dSig = [K~^T ; K2~^T] V (the two 64 x 64 states as the row halves of one M = 128 product).  The
// carry is read as stored, transposed or symmetrised.  The queries, keys and values (and the
// extra and partial tiles) have two slots each: chunk j's loads go into slot j % 2 as soon as
// chunk j - 2 has released it.  One pair (the two-operand-slot order): one G region, Y, the A
// operands, K~ and Sig0 in two slots by chunk parity; the epilogue runs EPI-1(j+1), EPI-S(j),
// EPI-Y(j).  Stacked pairs (one operand slot): G and then Y in one tensor-memory region,
// double-buffered by chunk parity; EPI-S(j), EPI-1(j+1), EPI-Y(j).  Swapped pair: one slot of
// everything; EPI-S(j), EPI-Y(j), EPI-1(j+1).
//
// A summary kernel forms the segment summaries (no chain) the same way.  Roles, bounded waits
// and one CTA per SM as in fo_tc.cu.
#include "fo_common.cuh"

namespace hla2 {

namespace {

namespace f64 {

constexpr int kW = 128, kD = 64;
constexpr int kThreads = 288;
// the output kernel: warp 0 issues the MMAs (and, except in the two-operand-slot order, the tile
// loads and stores), warps 1..8 are the epilogue, warp 9 issues the loads and stores in that order
constexpr int kThreadsOut = 320, kLoadWarp = 9;
constexpr uint32_t kTile = 128 * 128;  // a [128][64] bf16 tile: one SW128 block (16 KB)
constexpr uint32_t kSig = 64 * 128;    // the [64][64] bf16 state (8 KB)
constexpr uint32_t kTmemCols = 512;

// TWOA: the scaled keys K~ and the bf16 state Sig0 have two slots as well (by chunk parity).
// ST: the second pair's queries and keys (two slots each), its scaled keys beside K~ (the A
// operand of the M = 128 state product), and the [128][64] stacked bf16 state.
template <bool R2, bool KVS, bool XVS, bool ADD, bool TWOA = false, bool ST = false>
struct OutLayout {
    static constexpr uint32_t oX = 0;                                   // 2 slots
    static constexpr uint32_t oK = oX + 2 * kTile;                      // 2 slots
    static constexpr uint32_t oV = KVS ? oK : oK + 2 * kTile;           // 2 slots (KVS: the key slots)
    static constexpr uint32_t oE0 = (KVS ? oK : oV) + 2 * kTile;
    static constexpr uint32_t oXV = XVS ? oE0 : oV;                     // 2 slots
    static constexpr uint32_t oAD = XVS ? oXV + 2 * kTile : oE0;        // 2 slots
    static constexpr uint32_t oX2 = ADD ? oAD + 2 * kTile : oAD;        // ST: 2 slots
    static constexpr uint32_t oK2 = oX2 + 2 * kTile;                    // ST: 2 slots
    static constexpr uint32_t oKt = ST ? oK2 + 2 * kTile : oX2;         // K~ (TWOA: 2 slots; V~ / K2~ next)
    static constexpr uint32_t oKt2 = oKt + kTile;
    static constexpr uint32_t oST = (R2 || ST) ? oKt2 + kTile : oKt + (TWOA ? 2 : 1) * kTile;  // output tile
    static constexpr bool kTwoST = TWOA && !ADD;                        // (2 slots where they fit)
    static constexpr uint32_t oS0 = oST + (kTwoST ? 2 : 1) * kTile;     // bf16 Sig0 (TWOA: 2 slots)
    static constexpr uint32_t oGP = oS0 + ((TWOA || ST) ? 2 : 1) * kSig;  // g^0 .. g^(2W)
    static constexpr uint32_t oBar = oGP + 1088;
    static constexpr uint32_t oMisc = oBar + 24 * 8;
    static constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
    __host__ __device__ static constexpr uint32_t x(int j) { return oX + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t key(int j) { return oK + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t val(int j) { return KVS ? key(j) : oV + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t xv(int j) { return XVS ? oXV + (uint32_t)(j & 1) * kTile : val(j); }
    __host__ __device__ static constexpr uint32_t ad(int j) { return oAD + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t x2(int j) { return oX2 + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t k2(int j) { return oK2 + (uint32_t)(j & 1) * kTile; }
    __host__ __device__ static constexpr uint32_t kt(int j) { return oKt + (TWOA ? (uint32_t)(j & 1) * kTile : 0u); }
    __host__ __device__ static constexpr uint32_t s0(int j) { return oS0 + (TWOA ? (uint32_t)(j & 1) * kSig : 0u); }
    __host__ __device__ static constexpr uint32_t st(int j) { return oST + (kTwoST ? (uint32_t)(j & 1) * kTile : 0u); }
};

// Tensor-memory columns.  One pair (kTwoA, the two-slot order): G [0,128); Y of chunk j in
// [128,192) or [192,256) (with a next summary: Y [128,192), the summary [192,256)); A operands
// of chunk j in [256,352) or [352,448) (G~ 64 | fX 32); dSig [448,512).  Swapped pair: G1
// [0,128), G2 [128,256); after EPI-1 Y [0,64) and dSig [128,192); A operands [256,416)
// (G~1 | G~2 | fX).  Stacked pairs (ST, one operand slot): G and then Y of chunk j in [0,128)
// or [384,512) by chunk parity; dSig [128,192) over all 128 lanes (the two states); A operands
// [256,384) (G~ | fX | fX2).
template <bool R2, bool NSUM, bool ST = false>
struct Cols {
    static constexpr bool kTwoG = !R2;
    static constexpr bool kTwoA = !R2 && !ST;
    static constexpr bool kTwoY = kTwoA && !NSUM;
    static constexpr uint32_t TS = (R2 || ST) ? 128 : 448;
    static constexpr uint32_t TN = 192;
    __device__ static constexpr uint32_t TG(int j) { return kTwoG && !kTwoA && (j & 1) ? 384u : 0u; }
    __device__ static constexpr uint32_t TY(int j) { return kTwoA ? 128u + (kTwoY ? 64u * (uint32_t)(j & 1) : 0u) : TG(j); }
    __device__ static constexpr uint32_t TA(int j) { return kTwoA && (j & 1) ? 352u : 256u; }
    __device__ static constexpr uint32_t TX(int j) { return TA(j) + (R2 ? 128u : 64u); }
};

// BYT1 / BSF1: with two output stage slots, BYT / BSF serve even chunks and these odd ones;
// BGT1 / BSU1 likewise in the two-operand-slot order, where two threads wait on them
enum Bar { FX0 = 0, FX1, FK0, FK1, FV0, FV1, BG, BGT, BSU, BS, BYT, BN, BSF, BSF1, BYT1, BGT1, BSU1, kBarCount };

struct Maps {
    CUtensorMap x, k, v, xv, ad, out, x2, k2;
};

}  // namespace f64

// ----------------------------------------------------------------------------------------
template <bool REV, bool NSUM, bool R2, bool KVS, bool XVS, bool ADD, bool ST = false>
__global__ void __launch_bounds__(f64::kThreadsOut, 1)
    fo64_out_tc_kernel(const __grid_constant__ f64::Maps maps, const FoArgs a) {
    using C = f64::Cols<R2, NSUM, ST>;
    constexpr bool kTwoG = C::kTwoG, kTwoA = C::kTwoA;
    using Lay = f64::OutLayout<R2, KVS, XVS, ADD, kTwoA, ST>;
    static_assert(!ST || (!NSUM && !R2 && !KVS && !XVS && !ADD), "stacked pairs: plain values, one output");
    static_assert(Lay::kSmemBytes <= 232448, "shared memory of one CTA");
    constexpr int kW = f64::kW, kD = f64::kD;
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gp = reinterpret_cast<float*>(sm + Lay::oGP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Lay::oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::oMisc + 4);
    int* status = a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const FoSeg sg = la_seg(a, seg);
    const int nit = sg.nit;
    const float gam = head_decay(a.gamma, bh, a.H);
    const float log2g = (float)a.pow * log2f(gam);
    const float log2gn = (float)a.pow_next * log2f(gam);
    const float g = exp2f(log2g);

    for (int i = tid; i < 2 * kW + 1; i += f64::kThreadsOut) gp[i] = pow_decay(log2g, (float)i);
    if (tid == 0) {
        for (int b = 0; b < f64::kBarCount; ++b) {
            const bool from_epilogue = b == f64::BGT || b == f64::BGT1 || b == f64::BS || b == f64::BYT || b == f64::BYT1;
            tc::mbar_init(&bars[b], from_epilogue ? 8 : 1);
        }
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();

    // epilogue thread: TMEM lane / token row r, column half h: tile columns 32h .. 32h+31
    // (chunks 4h .. 4h+3); state row sr = r % 64, columns sc .. sc+15 (ST: stacked state row r,
    // columns 32h .. 32h+31)
    const int q4 = warp & 3, h = (warp - 1) >> 2;
    const int r = 32 * q4 + lane;
    const int sr = ST ? r : r & 63, sc = ST ? 32 * h : 32 * h + 16 * (r >> 6);
    constexpr int kSigN = ST ? 32 : 16;
    float sig[kSigN];
    auto publish_sig = [&](int jn) {  // Sig0 of chunk jn
#pragma unroll
        for (int j = 0; j < kSigN / 8; ++j)
            *reinterpret_cast<uint4*>(sm + Lay::s0(jn) + tc::sw128_chunk(sr, sc / 8 + j)) = la_pack8(&sig[8 * j]);
    };

    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, f64::kTmemCols);
    } else if (warp <= 8) {
        // (ST: rows 0..63 of the stacked state carry the first pair, rows 64..127 the second)
        const bool second = ST && r >= 64;
        const float* carry = second ? a.carry2 : a.carry;
        const int mode = second ? a.carry_mode2 : a.carry_mode, cr = sr & 63;
        if (carry && HLA2_IN(bh < a.BH && seg < a.nseg, 851)) {
            const float* src = carry + ((size_t)bh * a.nseg + seg) * kD * kD;
#pragma unroll
            for (int j = 0; j < kSigN; ++j) {
                const float x = src[(size_t)cr * kD + sc + j], xt = src[(size_t)(sc + j) * kD + cr];
                sig[j] = mode == 0 ? x : (mode == 1 ? xt : x + xt);
            }
        } else {
#pragma unroll
            for (int j = 0; j < kSigN; ++j) sig[j] = 0.f;
        }
        publish_sig(0);
        tc::fence_proxy_async();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    auto chunk_of = [&](int it) { return REV ? sg.c_end - 1 - it : sg.c_begin + it; };
    auto fx = [&](int j) { return &bars[(j & 1) ? f64::FX1 : f64::FX0]; };
    auto fk = [&](int j) { return &bars[(j & 1) ? f64::FK1 : f64::FK0]; };
    auto fv = [&](int j) { return &bars[(j & 1) ? f64::FV1 : f64::FV0]; };
    constexpr int kVTiles = (KVS ? 0 : 1) + (XVS ? 1 : 0) + (ADD ? 1 : 0);

    // the barriers that complete once per chunk and have two waiters in the two-operand-slot
    // order come in pairs by chunk parity, so that no wait can see a later phase
    auto bgt = [&](int j) { return &bars[kTwoA && (j & 1) ? f64::BGT1 : f64::BGT]; };
    auto bsu = [&](int j) { return &bars[kTwoA && (j & 1) ? f64::BSU1 : f64::BSU]; };
    auto par = [&](int j) { return (uint32_t)(kTwoA ? (j >> 1) & 1 : j & 1); };

    if (warp == 0 || warp == f64::kLoadWarp) {
        // ------------------------------------------------------------ control threads
        const bool mma_role = warp == 0;
        if (lane == 0 && nit > 0 && (kTwoA || mma_role)) {
            auto load1 = [&](uint32_t slot, const CUtensorMap* m, int c, uint64_t* bar) {
                tc::tma_load_3d(sm + slot, m, 0, c * kW, bh, bar);
            };
            // (ST: the second pair's tile comes with each, on the same barrier)
            auto load_x = [&](int j) {
                tc::mbar_arrive_expect_tx(fx(j), (ST ? 2 : 1) * f64::kTile);
                load1(Lay::x(j), &maps.x, chunk_of(j), fx(j));
                if (ST) load1(Lay::x2(j), &maps.x2, chunk_of(j), fx(j));
            };
            auto load_k = [&](int j) {
                tc::mbar_arrive_expect_tx(fk(j), (ST ? 2 : 1) * f64::kTile);
                load1(Lay::key(j), &maps.k, chunk_of(j), fk(j));
                if (ST) load1(Lay::k2(j), &maps.k2, chunk_of(j), fk(j));
            };
            auto load_v = [&](int j) {
                if (kVTiles == 0) return;
                tc::mbar_arrive_expect_tx(fv(j), kVTiles * f64::kTile);
                if (!KVS) load1(Lay::val(j), &maps.v, chunk_of(j), fv(j));
                if (XVS) load1(Lay::xv(j), &maps.xv, chunk_of(j), fv(j));
                if (ADD) load1(Lay::ad(j), &maps.ad, chunk_of(j), fv(j));
            };
            constexpr bool v_late = NSUM || ADD;  // the value group is still read after the products
            const uint32_t sKt2 = smem_u32(sm + Lay::oKt2), sST = smem_u32(sm + Lay::oST);
            constexpr uint32_t I_G = tc::idesc_bf16(128, 128, 0, 0);   // X K^T, K = 64 features
            constexpr uint32_t I_Y = tc::idesc_bf16(128, 64, 0, 1);    // A (TMEM) x MN-major B, N = 64
            constexpr uint32_t I_S = tc::idesc_bf16(128, 64, 1, 1);    // [A^T ; A^T] B, N = 64
            auto kdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 32u * ks, 16, 1024); };
            auto mdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 2048u * ks, 0, 1024); };
            int lx = 0, lk = 0, lv = 0;
            // a descriptor's address field counts 16-byte units: a K step of 32 bytes (K-major) is
            // +2, one of 2048 bytes (MN-major, 8 K-rows of a SW128 tile) is +128
            auto mma_g = [&](int j) {
                const uint32_t sX = smem_u32(sm + Lay::x(j)), sK = smem_u32(sm + Lay::key(j));
                const uint64_t dX = kdesc(sX, 0), dK = kdesc(sK, 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::mma_ss(tmem + C::TG(j), dX + 2u * ks, dK + 2u * ks, I_G, ks > 0);
                if (R2) {
                    const uint32_t sV = smem_u32(sm + Lay::val(j));
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + C::TG(j) + 128, kdesc(sX, ks), kdesc(sV, ks), I_G, ks > 0);
                }
                if (ST) {  // G += X2 K2^T
                    const uint32_t sX2 = smem_u32(sm + Lay::x2(j)), sK2 = smem_u32(sm + Lay::k2(j));
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_ss(tmem + C::TG(j), kdesc(sX2, ks), kdesc(sK2, ks), I_G, 1);
                }
                tc::mma_commit(&bars[f64::BG]);
            };
            auto wait_g_inputs = [&](int j) {
                tc::mbar_wait(fx(j), (j >> 1) & 1, abort, status, 131);
                tc::mbar_wait(fk(j), (j >> 1) & 1, abort, status, 132);
                if (R2) tc::mbar_wait(fv(j), (j >> 1) & 1, abort, status, 133);
                tc::fence_after_sync();
            };
            // after EPI-Y(j): the tile store and the next summary's products (finish_store), then,
            // once the next Gram is issued, the late loads and the stage freed (finish_release)
            auto finish_store = [&](int j) {
                if (Lay::kTwoST)
                    tc::mbar_wait(&bars[(j & 1) ? f64::BYT1 : f64::BYT], (j >> 1) & 1, abort, status, 138);
                else
                    tc::mbar_wait(&bars[f64::BYT], j & 1, abort, status, 138);
                tc::fence_after_sync();
                tc::tma_store_3d(&maps.out, sm + Lay::st(j), 0, chunk_of(j) * kW, bh);
                tc::bulk_commit();
                if (NSUM) {  // next summary: T_N += [Y^T ; Y^T] (w' U)
                    const uint32_t sXV = smem_u32(sm + Lay::xv(j)), sSTj = smem_u32(sm + Lay::st(j));
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ss(tmem + C::TN, mdesc(sSTj, ks), mdesc(sXV, ks), I_S, (j > 0 || ks > 0) ? 1u : 0u);
                    tc::mma_commit(&bars[f64::BN]);
                }
            };
            auto finish_release = [&](int j) {
                if (NSUM) tc::mbar_wait(&bars[f64::BN], j & 1, abort, status, 139);
                if (v_late && j + 2 < nit && kVTiles > 0) {  // slot j % 2 of the value group is free
                    load_v(j + 2);
                    ++lv;
                }
                if (Lay::kTwoST) {  // two stage slots: chunk j - 1's store has read its slot
                    tc::bulk_wait_read_but_last();
                    if (j > 0) tc::mbar_arrive(&bars[(j & 1) ? f64::BSF : f64::BSF1]);
                } else {
                    tc::bulk_wait_read_all();
                    tc::mbar_arrive(&bars[f64::BSF]);
                }
            };
            auto finish = [&](int j) {
                finish_store(j);
                finish_release(j);
            };

            auto prologue_loads = [&]() {  // chunks 0 and 1 in flight
                for (int j = 0; j < 2 && j < nit; ++j) {
                    load_x(j);
                    load_k(j);
                    ++lx;
                    ++lk;
                    if (kVTiles > 0) {
                        load_v(j);
                        ++lv;
                    }
                }
            };
            if constexpr (kTwoA) {
                // G in one region, read by EPI-1(j) before the next Gram; Y, the A operands, K~ and
                // Sig0 by chunk parity.  The epilogue runs EPI-1(j+1), EPI-S(j), EPI-Y(j): every
                // product of chunk j is issued as soon as EPI-1(j) and EPI-S(j-1) have arrived.
                // Warp 0 issues the MMAs, warp 9 the loads (the tiles three chunks ahead are
                // brought into L2 first, so that the loads two ahead are short) and the stores.
                if (mma_role) {
                    wait_g_inputs(0);
                    mma_g(0);
                    for (int j = 0; j < nit; ++j) {
                        tc::mbar_wait(bgt(j), par(j), abort, status, 134);  // G read; G~, fX, K~ written
                        if (j + 1 < nit) {
                            wait_g_inputs(j + 1);
                            mma_g(j + 1);
                        }
                        if (j > 0) tc::mbar_wait(&bars[f64::BS], (j - 1) & 1, abort, status, 136);  // Sig0 of chunk j
                        if (!KVS) tc::mbar_wait(fv(j), (j >> 1) & 1, abort, status, 135);
                        if (!C::kTwoY && j > 0)  // one Y region: EPI-Y(j - 1) has read it
                            tc::mbar_wait(&bars[(j & 1) ? f64::BYT : f64::BYT1], ((j - 1) >> 1) & 1, abort, status, 130);
                        tc::fence_after_sync();
                        const uint64_t dV = mdesc(smem_u32(sm + Lay::val(j)), 0);
                        const uint64_t dKt = mdesc(smem_u32(sm + Lay::kt(j)), 0);
                        const uint64_t dS0 = mdesc(smem_u32(sm + Lay::s0(j)), 0);
                        const uint32_t tY = tmem + C::TY(j), tA = tmem + C::TA(j), tX = tmem + C::TX(j);
                        // MMA-Y: Y = [G~ | fX] [V ; Sig0];  MMA-S: dSig = [K~^T ; K~^T] V
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) tc::mma_ts(tY, tA + 8 * ks, dV + 128u * ks, I_Y, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) tc::mma_ts(tY, tX + 8 * ks, dS0 + 128u * ks, I_Y, 1);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::mma_ss(tmem + C::TS, dKt + 128u * ks, dV + 128u * ks, I_S, ks > 0);
                        tc::mma_commit(bsu(j));
                    }
                    volatile int never = 0;  // drain (bounded, ignoring the abort flag)
                    tc::mbar_wait(bsu(nit - 1), par(nit - 1), &never, nullptr, 0);
                } else {
                    auto prefetch = [&](int j) {
                        const int c = chunk_of(j) * kW;
                        tc::tma_prefetch_3d(&maps.x, 0, c, bh);
                        tc::tma_prefetch_3d(&maps.k, 0, c, bh);
                        if (!KVS) tc::tma_prefetch_3d(&maps.v, 0, c, bh);
                        if (XVS) tc::tma_prefetch_3d(&maps.xv, 0, c, bh);
                        if (ADD) tc::tma_prefetch_3d(&maps.ad, 0, c, bh);
                    };
                    prologue_loads();
                    if (nit > 2) prefetch(2);
                    for (int j = 0; j < nit; ++j) {
                        tc::mbar_wait(bgt(j), par(j), abort, status, 139);  // MMA-G(j) and EPI-1(j) done
                        if (j + 3 < nit) prefetch(j + 3);
                        if (j + 2 < nit) {  // X and key slots j % 2 are free
                            load_x(j + 2);
                            ++lx;
                            if (!KVS) {
                                load_k(j + 2);
                                ++lk;
                            }
                        }
                        if (j > 0) finish(j - 1);  // after EPI-Y(j - 1)
                        tc::mbar_wait(bsu(j), par(j), abort, status, 137);  // chunk j's products done
                        if (j + 2 < nit) {  // the value slot j % 2 is free (keys as values: the key slot)
                            if (KVS) {
                                load_k(j + 2);
                                ++lk;
                            }
                            if (!v_late && !KVS) {
                                load_v(j + 2);
                                ++lv;
                            }
                        }
                    }
                    finish(nit - 1);
                }
            } else {
            prologue_loads();
            wait_g_inputs(0);
            mma_g(0);
            for (int j = 0; j < nit; ++j) {
                tc::mbar_wait(&bars[f64::BGT], j & 1, abort, status, 134);  // G read; G~, fX, K~ written
                if (j > 0) tc::mbar_wait(&bars[f64::BS], (j - 1) & 1, abort, status, 136);  // Sig0 of chunk j
                if (j + 2 < nit) {  // X slot j % 2 is free (and key slot j % 2, unless MMA-Y reads it)
                    load_x(j + 2);
                    ++lx;
                    if (!R2 && !KVS) {
                        load_k(j + 2);
                        ++lk;
                    }
                }
                if (!KVS) tc::mbar_wait(fv(j), (j >> 1) & 1, abort, status, 135);
                tc::fence_after_sync();
                const uint32_t sK = smem_u32(sm + Lay::key(j)), sV = smem_u32(sm + Lay::val(j));
                const uint32_t sKt = smem_u32(sm + Lay::kt(j)), sS0 = smem_u32(sm + Lay::s0(j));
                // MMA-Y: Y = [G~ | (G~2) | fX (| fX2)] [V ; (K) ; Sig0 (; Sig0_2)]
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ts(tmem + C::TY(j), tmem + C::TA(j) + 8 * ks, mdesc(sV, ks), I_Y, ks > 0);
                if (R2)
                    for (int ks = 0; ks < 8; ++ks)
                        tc::mma_ts(tmem + C::TY(j), tmem + C::TA(j) + 64 + 8 * ks, mdesc(sK, ks), I_Y, 1);
                for (int ks = 0; ks < (ST ? 8 : 4); ++ks)
                    tc::mma_ts(tmem + C::TY(j), tmem + C::TX(j) + 8 * ks, mdesc(sS0, ks), I_Y, 1);
                // MMA-S: dSig = [K~^T ; K~^T] V (R2: + [V~^T ; V~^T] K; ST: [K~^T ; K2~^T] V, the
                // second row half read one tile on)
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem + C::TS, ST ? tc::smem_desc(sKt + 2048u * ks, f64::kTile, 1024) : mdesc(sKt, ks),
                               mdesc(sV, ks), I_S, ks > 0);
                if (R2)
                    for (int ks = 0; ks < 8; ++ks) tc::mma_ss(tmem + C::TS, mdesc(sKt2, ks), mdesc(sK, ks), I_S, 1);
                tc::mma_commit(&bars[f64::BSU]);
                if (kTwoG) {
                    // EPI-Y(j - 1) has read G / Y region (j + 1) % 2: the next Gram goes before the
                    // wait for the previous tile store to leave the stage
                    if (j > 0) finish_store(j - 1);
                    if (j + 1 < nit) {
                        wait_g_inputs(j + 1);
                        mma_g(j + 1);
                    }
                    if (j > 0) finish_release(j - 1);
                    tc::mbar_wait(&bars[f64::BSU], j & 1, abort, status, 137);  // chunk j's products done
                } else {
                    finish(j);  // after EPI-Y(j): chunk j's products are done
                }
                if (j + 2 < nit) {  // key slot j % 2 is free (and the value slot, without late reads)
                    if (R2 || KVS) {  // MMA-Y reads the raw keys (the swapped pair, or keys as values)
                        load_k(j + 2);
                        ++lk;
                    }
                    if (!v_late && !KVS) {
                        load_v(j + 2);
                        ++lv;
                    }
                }
                if (!kTwoG && j + 1 < nit) {
                    wait_g_inputs(j + 1);
                    mma_g(j + 1);
                }
            }
            if (kTwoG) finish(nit - 1);
            }
            volatile int never = 0;
            if (!kTwoA) tc::mbar_wait(&bars[f64::BSU], (nit - 1) & 1, &never, nullptr, 0);
            if (NSUM) tc::mbar_wait(&bars[f64::BN], (nit - 1) & 1, &never, nullptr, 0);
            // every load group's last phase, per slot
            auto drain = [&](int count, uint64_t* b0, uint64_t* b1) {
                if (count > 0) tc::mbar_wait(b0, ((count + 1) / 2 - 1) & 1, &never, nullptr, 0);
                if (count > 1) tc::mbar_wait(b1, (count / 2 - 1) & 1, &never, nullptr, 0);
            };
            drain(lx, &bars[f64::FX0], &bars[f64::FX1]);
            drain(lk, &bars[f64::FK0], &bars[f64::FK1]);
            drain(lv, &bars[f64::FV0], &bars[f64::FV1]);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int row0 = 32 * q4;
        const uint32_t lrow = tmem + ((uint32_t)row0 << 16);
        const float ginv = g > 0.f ? 1.f / g : 0.f;

        auto epi1 = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            const bool live = r < Wc;
            unsigned char* sX = sm + Lay::x(j);
            unsigned char* sK = sm + Lay::key(j);
            unsigned char* sV = sm + Lay::val(j);
            tc::mbar_wait(fx(j), (j >> 1) & 1, abort, status, 141);
            tc::mbar_wait(fk(j), (j >> 1) & 1, abort, status, 142);
            if (R2) tc::mbar_wait(fv(j), (j >> 1) & 1, abort, status, 143);
            tc::mbar_wait(&bars[f64::BG], j & 1, abort, status, 144);
            tc::fence_after_sync();
#pragma unroll
            for (int gi = 0; gi < (R2 ? 2 : 1); ++gi) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int cb = 64 * h + 32 * p;
                    uint32_t pk[16];
                    la_masked_pack<REV>(lrow + C::TG(j) + 128 * gi + cb, r, cb, row0, log2g, g, ginv, pk);
                    tc::tmem_st16(lrow + C::TA(j) + 64 * gi + cb / 2, pk);
                }
            }
            // fX: this thread's 32 features of row r -> 16 packed columns (ST: fX2 32 columns on)
#pragma unroll
            for (int xi = 0; xi < (ST ? 2 : 1); ++xi) {
                const unsigned char* sXi = xi == 0 ? sX : sm + Lay::x2(j);
                const float f = live ? (REV ? gp[Wc - r] : gp[r + 1]) : 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 x = la_scale_chunk(*reinterpret_cast<const uint4*>(sXi + tc::sw128_chunk(r, 4 * h + i)), f);
                    pk[4 * i] = x.x, pk[4 * i + 1] = x.y, pk[4 * i + 2] = x.z, pk[4 * i + 3] = x.w;
                }
                tc::tmem_st16(lrow + C::TX(j) + 32 * xi + 16 * h, pk);
            }
            const float w = live ? (REV ? gp[r] : gp[Wc - 1 - r]) : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = tc::sw128_chunk(r, 4 * h + i);
                *reinterpret_cast<uint4*>(sm + Lay::kt(j) + off) = la_scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w);
                if (R2 || ST)  // V~ (swapped pair) or K2~ (stacked pairs)
                    *reinterpret_cast<uint4*>(sm + Lay::oKt2 + off) =
                        la_scale_chunk(*reinterpret_cast<const uint4*>((ST ? sm + Lay::k2(j) : sV) + off), w);
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bgt(j));
        };

        auto epis = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            tc::mbar_wait(bsu(j), par(j), abort, status, 145);
            tc::fence_after_sync();
            const float rho = gp[Wc];
#pragma unroll
            for (int part = 0; part < kSigN / 16; ++part) {
                uint32_t v[16];
                tc::tmem_ld16(lrow + C::TS + sc + 16 * part, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) sig[16 * part + i] = rho * sig[16 * part + i] + __uint_as_float(v[i]);
            }
            if (j + 1 < nit) publish_sig(j + 1);  // the products that read this slot last have completed
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[f64::BS]);
        };

        auto epiy = [&](int j) {
            const int c = chunk_of(j);
            const int Wc = min(kW, a.n - c * kW);
            const bool live = r < Wc;
            if (Lay::kTwoST) {  // the stage slot j % 2 was last stored from by chunk j - 2 (released
                                // once chunk j - 1's store is issued)
                if (j > 1) tc::mbar_wait(&bars[(j & 1) ? f64::BSF1 : f64::BSF], ((j >> 1) - 1) & 1, abort, status, 146);
            } else if (j > 0) {
                tc::mbar_wait(&bars[f64::BSF], (j - 1) & 1, abort, status, 146);
            }
            if (ADD || (NSUM && XVS)) tc::mbar_wait(fv(j), (j >> 1) & 1, abort, status, 147);
            tc::fence_after_sync();
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t v[16];
                tc::tmem_ld16(lrow + C::TY(j) + 32 * h + 16 * p, v);
                tc::tmem_wait_ld();
                float y[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) y[i] = __uint_as_float(v[i]);
                if (ADD) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 x = *reinterpret_cast<const uint4*>(sm + Lay::ad(j) + tc::sw128_chunk(r, 4 * h + 2 * p + i));
                        y[8 * i + 0] += la_bf_lo(x.x), y[8 * i + 1] += la_bf_hi(x.x);
                        y[8 * i + 2] += la_bf_lo(x.y), y[8 * i + 3] += la_bf_hi(x.y);
                        y[8 * i + 4] += la_bf_lo(x.z), y[8 * i + 5] += la_bf_hi(x.z);
                        y[8 * i + 6] += la_bf_lo(x.w), y[8 * i + 7] += la_bf_hi(x.w);
                    }
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    *reinterpret_cast<uint4*>(sm + Lay::st(j) + tc::sw128_chunk(r, 4 * h + 2 * p + i)) = la_pack8(&y[8 * i]);
            }
            if (NSUM) {
                const int pos = (c - sg.c_begin) * kW + r;
                const float wn = live ? pow_decay(log2gn, (float)(REV ? pos : sg.L - 1 - pos)) : 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = Lay::xv(j) + tc::sw128_chunk(r, 4 * h + i);
                    *reinterpret_cast<uint4*>(sm + off) = la_scale_chunk(*reinterpret_cast<const uint4*>(sm + off), wn);
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[Lay::kTwoST && (j & 1) ? f64::BYT1 : f64::BYT]);
        };

        if (nit > 0) epi1(0);
        for (int j = 0; j < nit; ++j) {
            if (kTwoA) {
                if (j + 1 < nit) epi1(j + 1);
                epis(j);
                epiy(j);
            } else if (kTwoG) {
                epis(j);
                if (j + 1 < nit) epi1(j + 1);
                epiy(j);
            } else {
                epis(j);
                epiy(j);
                if (j + 1 < nit) epi1(j + 1);
            }
        }
        if (NSUM && nit > 0 && HLA2_IN(bh < a.BH && seg < a.nseg, 852)) {
            tc::mbar_wait(&bars[f64::BN], (nit - 1) & 1, abort, status, 148);
            tc::fence_after_sync();
            uint32_t v[16];
            tc::tmem_ld16(lrow + C::TN + sc, v);
            tc::tmem_wait_ld();
            float* dst = a.summary + ((size_t)bh * a.nseg + seg) * kD * kD + (size_t)sr * kD + sc;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                  __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, f64::kTmemCols);
}

// ----------------------------------------------------------------------------------------
// Summary kernel: Sig_B[s] = sum_{i in s} w_i k_i v_i^T (forward: decayed to the segment's end;
// reverse: to its start), two stages, [K~^T ; K~^T] V accumulated in tensor memory.
namespace f64s {
template <bool KVS>
struct Layout {
    static constexpr uint32_t oK = 0;                                     // 2 stages
    static constexpr uint32_t oV = KVS ? oK : oK + 2 * f64::kTile;        // 2 stages
    static constexpr uint32_t oKt = (KVS ? oK : oV) + 2 * f64::kTile;     // 2 stages
    static constexpr uint32_t oBar = oKt + 2 * f64::kTile;
    static constexpr uint32_t oMisc = oBar + 16 * 8;
    static constexpr uint32_t kSmemBytes = oMisc + 16 + 1024;
};
enum Bar { F0 = 0, F1, T0, T1, N0, N1, kBarCount };
}  // namespace f64s

template <bool REV, bool KVS>
__global__ void __launch_bounds__(f64::kThreads, 1)
    fo64_sum_tc_kernel(const __grid_constant__ f64::Maps maps, const FoArgs a) {
    using Lay = f64s::Layout<KVS>;
    constexpr int kW = f64::kW, kD = f64::kD;
    pdl_trigger();
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::oBar);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + Lay::oMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + Lay::oMisc + 4);
    int* status = a.status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const FoSeg sg = la_seg(a, seg);
    const int nit = sg.nit;
    const float log2g = (float)a.pow * log2f(head_decay(a.gamma, bh, a.H));

    if (tid == 0) {
        for (int b = 0; b < f64s::kBarCount; ++b) tc::mbar_init(&bars[b], (b == f64s::T0 || b == f64s::T1) ? 8 : 1);
        *abort = 0;
        tc::mbar_fence_init();
    }
    pdl_wait();
    if (warp == 0) tc::tmem_alloc(tmem_holder, 64);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    auto chunk_of = [&](int it) { return REV ? sg.c_end - 1 - it : sg.c_begin + it; };

    if (warp == 0) {
        if (lane == 0 && nit > 0) {
            auto load = [&](int it) {
                const int s = it & 1, c = chunk_of(it);
                uint64_t* bar = &bars[f64s::F0 + s];
                tc::mbar_arrive_expect_tx(bar, (KVS ? 1 : 2) * f64::kTile);
                tc::tma_load_3d(sm + Lay::oK + s * f64::kTile, &maps.k, 0, c * kW, bh, bar);
                if (!KVS) tc::tma_load_3d(sm + Lay::oV + s * f64::kTile, &maps.v, 0, c * kW, bh, bar);
            };
            constexpr uint32_t I_S = tc::idesc_bf16(128, 64, 1, 1);
            auto mdesc = [](uint32_t base, int ks) { return tc::smem_desc(base + 2048u * ks, 0, 1024); };
            load(0);
            if (nit > 1) load(1);
            for (int it = 0; it < nit; ++it) {
                const int s = it & 1;
                const uint32_t ph = (it >> 1) & 1;
                tc::mbar_wait(&bars[f64s::T0 + s], ph, abort, status, 151);
                tc::fence_after_sync();
                const uint32_t sKt = smem_u32(sm + Lay::oKt + s * f64::kTile);
                const uint32_t sV = smem_u32(sm + Lay::oV + s * f64::kTile);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_ss(tmem, mdesc(sKt, ks), mdesc(sV, ks), I_S, (it > 0 || ks > 0) ? 1u : 0u);
                tc::mma_commit(&bars[f64s::N0 + s]);
                if (it + 2 < nit) {
                    tc::mbar_wait(&bars[f64s::N0 + s], ph, abort, status, 152);
                    load(it + 2);
                }
            }
            volatile int never = 0;
            tc::mbar_wait(&bars[f64s::N0 + ((nit - 1) & 1)], ((nit - 1) >> 1) & 1, &never, nullptr, 0);
            if (nit > 1) tc::mbar_wait(&bars[f64s::N0 + ((nit - 2) & 1)], ((nit - 2) >> 1) & 1, &never, nullptr, 0);
        }
        __syncwarp();
    } else {
        const int q4 = warp & 3, h = (warp - 1) >> 2;
        const int r = 32 * q4 + lane;
        const int sr = r & 63, sc = 32 * h + 16 * (r >> 6);
        const uint32_t lrow = tmem + ((uint32_t)(32 * q4) << 16);
        for (int it = 0; it < nit; ++it) {
            const int s = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int c = chunk_of(it);
            const int Wc = min(kW, a.n - c * kW);
            tc::mbar_wait(&bars[f64s::F0 + s], ph, abort, status, 153);
            const int pos = (c - sg.c_begin) * kW + r;
            const float w = r < Wc ? pow_decay(log2g, (float)(REV ? pos : sg.L - 1 - pos)) : 0.f;
            unsigned char* sK = sm + Lay::oK + s * f64::kTile;
            unsigned char* sKt = sm + Lay::oKt + s * f64::kTile;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t off = tc::sw128_chunk(r, 4 * h + i);
                *reinterpret_cast<uint4*>(sKt + off) = la_scale_chunk(*reinterpret_cast<const uint4*>(sK + off), w);
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[f64s::T0 + s]);
        }
        if (nit > 0 && HLA2_IN(bh < a.BH && seg < a.nseg, 853)) {
            tc::mbar_wait(&bars[f64s::N0 + ((nit - 1) & 1)], ((nit - 1) >> 1) & 1, abort, status, 154);
            tc::fence_after_sync();
            uint32_t v[16];
            tc::tmem_ld16(lrow + sc, v);
            tc::tmem_wait_ld();
            float* dst = a.summary + ((size_t)bh * a.nseg + seg) * kD * kD + (size_t)sr * kD + sc;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                                  __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

template <typename K>
int f64_launch(K kfn, uint32_t smem, const f64::Maps& maps, const FoArgs& a, cudaStream_t st,
               int threads = f64::kThreads) {
    if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -1;
    if (launch_pdl(kfn, dim3(a.nseg, a.BH), dim3(threads), smem, st, maps, a) != cudaSuccess) return -1;
    return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

size_t fo64_tc_max_smem() {
    // the instantiated layouts: next summary over an extra tile (NSUM), plain (two slots for the
    // A-side operands), swapped pair, partial added (keys as values or not), next summary over
    // the values (NSUM), stacked pairs
    const uint32_t sizes[] = {f64::OutLayout<false, true, true, false, true>::kSmemBytes,
                              f64::OutLayout<false, false, false, false, true>::kSmemBytes,
                              f64::OutLayout<true, false, false, false>::kSmemBytes,
                              f64::OutLayout<false, true, false, true, true>::kSmemBytes,
                              f64::OutLayout<false, false, false, true, true>::kSmemBytes,
                              f64::OutLayout<false, false, true, false, true>::kSmemBytes,
                              f64::OutLayout<false, false, false, false, false, true>::kSmemBytes,
                              f64s::Layout<false>::kSmemBytes, f64s::Layout<true>::kSmemBytes};
    uint32_t m = 0;
    for (uint32_t x : sizes) m = x > m ? x : m;
    return m;
}

int launch_fo64_tc_summary(const FoArgs& a, const void* k, const void* v, bool reverse, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    f64::Maps m{};
    if (!la_map(&m.k, k, a.BH, a.n, 64) || !la_map(&m.v, v ? v : k, a.BH, a.n, 64)) return -2;
    const bool kvs = !v || v == k;
    if (kvs)
        return reverse ? f64_launch(fo64_sum_tc_kernel<true, true>, f64s::Layout<true>::kSmemBytes, m, a, st)
                       : f64_launch(fo64_sum_tc_kernel<false, true>, f64s::Layout<true>::kSmemBytes, m, a, st);
    return reverse ? f64_launch(fo64_sum_tc_kernel<true, false>, f64s::Layout<false>::kSmemBytes, m, a, st)
                   : f64_launch(fo64_sum_tc_kernel<false, false>, f64s::Layout<false>::kSmemBytes, m, a, st);
}

// As launch_fo_tc_out (fo_tc.cu), for d = dv = 64.
int launch_fo64_tc_out(const FoArgs& a, const void* x, const void* k, const void* v, bool r2, int next_sum,
                       const void* xv, const void* add, void* out, bool reverse, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    f64::Maps m{};
    const bool kvs = v == nullptr, nsum = next_sum != 0, xvs = next_sum == 2, addp = add != nullptr;
    if (!la_map(&m.x, x, a.BH, a.n, 64) || !la_map(&m.k, k, a.BH, a.n, 64) ||
        !la_map(&m.v, kvs ? k : v, a.BH, a.n, 64) || !la_map(&m.out, out, a.BH, a.n, 64))
        return -2;
    if (xvs && !la_map(&m.xv, xv, a.BH, a.n, 64)) return -2;
    if (addp && !la_map(&m.ad, add, a.BH, a.n, 64)) return -2;
    if (nsum && !a.summary) return -2;
#define HLA2_F64(REV, NSUM, R2, KVS, XVS, ADD)                                                               \
    if (reverse == REV && nsum == NSUM && r2 == R2 && kvs == KVS && xvs == XVS && addp == ADD)              \
        return f64_launch(fo64_out_tc_kernel<REV, NSUM, R2, KVS, XVS, ADD>,                                    \
                          f64::OutLayout<R2, KVS, XVS, ADD, f64::Cols<R2, NSUM>::kTwoA>::kSmemBytes, m, a, st, \
                          f64::kThreadsOut);
    HLA2_F64(false, true, false, true, true, false)    // p = LA(q, k, k), next summary over (p, v)
    HLA2_F64(false, false, false, true, false, false)   // p = LA(q, k, k) (the summary over (p, v) apart)
    HLA2_F64(false, false, false, false, false, false) // o = LA(q, p, v);  Z dO = LA(dO, v, p)
    HLA2_F64(true, true, false, false, false, false)   // dp = RLA(v, dO, q), next summary over (dp, q)
    HLA2_F64(true, false, false, false, false, false)  // dv = RLA(p, q, dO)
    HLA2_F64(true, false, true, false, false, false)   // dk = RLA(k, dp, q) + RLA(k, q, dp)
    HLA2_F64(false, false, false, true, false, true)   // dq = LA(dp, k, k) + Z dO
    // the AHLA reverse mode (u = LA(q, k, v), o = LA(q, k, u))
    HLA2_F64(false, true, false, false, true, false)   // u = LA(q, k, v), next summary over (u, k)
    HLA2_F64(true, true, false, false, true, false)    // du = RLA(k, q, dO), next summary over (du, q)
    HLA2_F64(true, false, false, false, false, true)   // dk = RLA(v, du, q) + RLA(u, dO, q)
    HLA2_F64(false, false, false, false, false, true)  // dq = LA(du, v, k) + LA(dO, u, k)
#undef HLA2_F64
    return -3;
}

int launch_fo64_tc_out2(const FoArgs& a, const void* x, const void* k, const void* x2, const void* k2, const void* v,
                        void* out, bool reverse, cudaStream_t st) {
    if (a.BH <= 0 || a.nseg <= 0) return 0;
    f64::Maps m{};
    if (!la_map(&m.x, x, a.BH, a.n, 64) || !la_map(&m.k, k, a.BH, a.n, 64) || !la_map(&m.x2, x2, a.BH, a.n, 64) ||
        !la_map(&m.k2, k2, a.BH, a.n, 64) || !la_map(&m.v, v, a.BH, a.n, 64) || !la_map(&m.out, out, a.BH, a.n, 64))
        return -2;
    constexpr uint32_t smem = f64::OutLayout<false, false, false, false, false, true>::kSmemBytes;
    // dk = RLA(u, dO, q) + RLA(v, du, q) (reverse);  dq = LA(dO, u, k) + LA(du, v, k) (forward)
    return reverse ? f64_launch(fo64_out_tc_kernel<true, false, false, false, false, false, true>, smem, m, a, st,
                                f64::kThreadsOut)
                   : f64_launch(fo64_out_tc_kernel<false, false, false, false, false, false, true>, smem, m, a, st,
                                f64::kThreadsOut);
}

}  // namespace hla2

HLA2_DEBUG_READER(fo64_tc)
