// Chunk-parallel main backward kernel: one CTA (8 warps) per (chunk, head).
//
// Given the chunk-start state S0 and the state gradient at the chunk end dS_C
// (both from the serial recurrences), every gradient of the chunk is local.
// Forward quantities are recomputed (chunk algebra of the gated delta rule,
// UT/WY form):
//   A  = strict_lower(diag(beta) kd' ki'^T),  P = lower(qd' ki'^T)
//   E  = V - kd S0,  Y = diag(beta) E,  u = T Y   (T = (I + A)^-1 from the prep kernel)
// and the reverse pass is, in order,
//   dqd  = dO S0^T                              du  = P^T dO + kr dS_C
//   dY   = T^T du,  dv = beta dY                dkd = -beta (dY S0^T)
//   dkr  = u dS_C^T                             dgT = e^{gT} rowsum(dS_C . S0) + colsum(dkr . kr)
//   dP   = lower(dO u^T)                        dA  = -strict_lower(dY u^T)
//   dqd' = dP ki',  dkd' = (beta dA) ki'        dki' = dP^T qd' + (beta dA)^T kd'
//   dlogit = (1 - beta) (<dY, beta E> + rowsum(dA . A))
// and the elementwise assembly of "FlashKDA之backward（K1）" (§3.2-§3.3, §5):
//   dqn = scale (dqd e^{gc} + dqd' e^{gc-ref})
//   dkn = dkd e^{gc} + dkd' e^{gc-ref} + dki' e^{ref-gc} + dkr e^{gT-gc}
//   dgc = qn dqn + kn (dkd e^{gc} + dkd' e^{gc-ref} - dki' e^{ref-gc} - dkr e^{gT-gc})
//   L2-norm backward of dqn, dkn; dg = reverse_cumsum(dgc) + dgT; the GDN
//   gate gradient is the channel sum, the KDA gate runs its chain rule and
//   reduces dA_log, ddt_bias with one atomic per CTA and channel.
// The per-element gradients w.r.t. qn and kn live in registers for the whole
// kernel: every C x D product uses the same warp tiling.
#include "gdr_chunk.cuh"

namespace gdr {

template <int D, bool KDA>
struct MainSmem {
    static constexpr int ROWB = 2 * D;
    static constexpr int TCD = CH * ROWB;
    static constexpr int TDD = D * ROWB;
    static constexpr int TCC = CH * 128;
    static constexpr int oK = 0, oV = oK + TCD, oDO = oV + TCD, oS0 = oDO + TCD, oDS = oS0 + TDD,
                         oT = oDS + TDD, oA = oT + TCC, oP = oA + TCC, oU = oP + TCC, oX1 = oU + TCD,
                         oX2 = oX1 + TCD, oG = oX2 + TCD, oSmall = oG + Gates<D, KDA>::floats() * 4;
    // small arrays (floats): invQ, invK, beta [C] each, fac[4][C], dgT partials [4][D] and [D],
    // dbeta partials [4][C], rowq[2][C], rowk[2][C], misc[64]
    static constexpr int nSmall = 3 * CH + 4 * CH + 5 * D + 4 * CH + 4 * CH + 64;
    static constexpr int oEnd = (oSmall + nSmall * 4 + 127) / 128 * 128;
    // Residual (lo) tiles of the precise mode.  They live on the state tiles once
    // those are dead (D = 128: S0 holds dP_lo, (beta dA)_lo, ki'_lo; dS holds
    // qd'_lo, kd'_lo); for D = 64 the last three get their own space.
    static constexpr bool BIG = (D == 128);
    static constexpr int oDPlo = oS0, oBDAlo = BIG ? oS0 + TCC : oDS, oKIlo = BIG ? oS0 + 2 * TCC : oEnd,
                         oQDlo = BIG ? oDS : oEnd + TCD, oKDlo = BIG ? oDS + TCD : oEnd + 2 * TCD;
    static constexpr int bytes = (BIG || !KDA) ? oEnd : oEnd + 3 * TCD;
    static_assert(2 * TDD >= CH * D * 4, "dgc scratch must fit in the state tiles");
};

template <int D, bool KDA>
__global__ void __launch_bounds__(256, 1) k_main(const Params p) {
    if (!states_header_ok(p)) {  // saved states of another variant or shape: write nothing
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, ST_STATES_MISMATCH);
        return;
    }
    using SM = MainSmem<D, KDA>;
    using TileCD = SwzTile<SM::ROWB>;
    using TileCC = SwzTile<128>;
    constexpr int NTD = D / 16;
    // KDA runs the precise mode: the operands that carry the per-channel gate
    // gradient (u and beta E, dP and beta dA, and the in-chunk tiles qd', kd',
    // ki' of the gradient products) are bf16 pairs hi + lo, each product
    // hi*hi + lo*hi + hi*lo, because dA_log and ddt_bias sum dg over every token.
    constexpr bool PREC = KDA;
    extern __shared__ __align__(1024) unsigned char smem[];

    const int chunk = blockIdx.x, h = blockIdx.y;
    ChunkInfo ci;
    if (!lookup_chunk(chunk, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, ci)) return;

    TileCD sK{smem + SM::oK}, sV{smem + SM::oV}, sDO{smem + SM::oDO}, sU{smem + SM::oU},
        sX1{smem + SM::oX1}, sX2{smem + SM::oX2};
    TileCD sS0{smem + SM::oS0}, sDS{smem + SM::oDS};  // D x D tiles, same row size
    TileCC sT{smem + SM::oT}, sA{smem + SM::oA}, sP{smem + SM::oP};
    TileCC sDPlo{smem + SM::oDPlo}, sBDAlo{smem + SM::oBDAlo};
    TileCD sKIlo{smem + SM::oKIlo}, sQDlo{smem + SM::oQDlo}, sKDlo{smem + SM::oKDlo};
    float* gbase = reinterpret_cast<float*>(smem + SM::oG);
    Gates<D, KDA> G;
    G.gc = gbase;
    G.ref = gbase + (KDA ? CH * G.LDG : CH);
    G.gT = G.ref + (KDA ? D : 1);
    float* sInvQ = reinterpret_cast<float*>(smem + SM::oSmall);
    float* sInvK = sInvQ + CH;
    float* sBeta = sInvK + CH;
    float* sFac = sBeta + CH;       // GDN per-row factors [4][C]
    // Partial sums with one writer per slot, summed in a fixed order (bitwise
    // reproducible): dgT from the kr product per 16-row band [4][D] and from the
    // state term [D]; dbeta per column half of the dY and dA products [4][C].
    float* sDgTp = sFac + 4 * CH;   // [4][D]
    float* sDgTs = sDgTp + 4 * D;   // [D]
    float* sDb = sDgTs + D;         // [4][C]
    float* sRowQ = sDb + 4 * CH;    // [2][C]
    float* sRowK = sRowQ + 2 * CH;  // [2][C]
    float* sMisc = sRowK + 2 * CH;  // [64]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t tdd = ((size_t)chunk * p.H + h) * D * D;
    const size_t tcc = ((size_t)chunk * p.H + h) * CH * CH;

    // ---- loads -------------------------------------------------------------
    const int hq = qk_head(p, h);  // q / k head of this value head
    async_load_rows<D>(sK, p.k, p, ci, hq, p.Hk);
    async_load_rows<D>(sV, p.v, p, ci, h);
    async_load_rows<D>(sDO, p.dO, p, ci, h);
    async_load_tile<D, D>(sS0, p.S0 + tdd);
    async_load_tile<D, D>(sDS, p.dS + tdd);
    async_load_tile<CH, CH>(sT, p.Tm + tcc);
    cp_async_commit();
    load_gates<D, KDA>(p, ci, h, G, false);
    load_beta(p, ci, h, sBeta);
    row_inv_norms_global<D>(p.q, p, ci, hq, sInvQ, p.Hk);
    cp_async_wait<0>();
    __syncthreads();
    row_inv_norms_smem<D>(sK, sInvK);
    if (!KDA) {
        for (int r = threadIdx.x; r < CH; r += blockDim.x) {
            sFac[0 * CH + r] = gate_factor<F_KD>(G, r, 0);
            sFac[1 * CH + r] = gate_factor<F_KDP>(G, r, 0);
            sFac[2 * CH + r] = gate_factor<F_KIP>(G, r, 0);
            sFac[3 * CH + r] = gate_factor<F_KR>(G, r, 0);
        }
    }
    // dgT (state part) = e^{gT} rowsum(dS_C . S0): the saved states are value-major
    // ([dv][dk]), so for each key channel d it is a column sum over the value rows
    {
        constexpr int NG = 256 / (D / 2);  // row groups per column pair
        const int cp = threadIdx.x / NG, g = threadIdx.x % NG;
        float s0 = 0.f, s1 = 0.f;
        for (int j = g; j < D; j += NG) {
            const float2 a = unpack_bf16(*reinterpret_cast<const uint32_t*>(sS0.ptr(j, 2 * cp)));
            const float2 b = unpack_bf16(*reinterpret_cast<const uint32_t*>(sDS.ptr(j, 2 * cp)));
            s0 += a.x * b.x;
            s1 += a.y * b.y;
        }
#pragma unroll
        for (int o = 1; o < NG; o <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (g == 0) {
            sDgTs[2 * cp] = s0 * __expf(G.gTv(2 * cp));
            sDgTs[2 * cp + 1] = s1 * __expf(G.gTv(2 * cp + 1));
        }
    }
    __syncthreads();

    auto fac = [&](int kind, int r, int d) -> float {
        if (!KDA) return sFac[kind * CH + r];
        switch (kind) {
            case F_KD: return gate_factor<F_KD>(G, r, d);
            case F_KDP: return gate_factor<F_KDP>(G, r, d);
            case F_KIP: return gate_factor<F_KIP>(G, r, d);
            default: return gate_factor<F_KR>(G, r, d);
        }
    };
    // value of a derived in-chunk tile element as the gradient products see it
    // (exact bf16 operand, or the fp32 value the hi + lo pair represents)
    auto tile_val = [&](float x, float m, float f) -> float {
        return PREC ? x * m * f : derived_val(x, m, f);
    };

    // warp tilings
    const int mC = 16 * (warp & 3), nC = 32 * (warp >> 2);       // C x C outputs: 16 x 32 per warp
    const int mD = 16 * (warp & 3), nD = (D / 2) * (warp >> 2);  // C x D outputs: 16 x D/2 per warp

    // Register accumulators over the C x D tile (same warp tiling for every
    // C x D product): gradients w.r.t. qn and kn, and dgc, the gradient w.r.t.
    // the cumulative gate.  dgc adds, for every derived tile X = base * e^{+-gc},
    // +-X * dX with X the value the tensor-core product consumed, so the paired
    // terms of each in-chunk product (row r, row s) cancel to fp32 rounding in the
    // reverse cumsum instead of to bf16 rounding.
    float dQn[1][NTD][4], dKn[1][NTD][4], dGc[1][NTD][4];
    zero_acc(dQn);
    zero_acc(dKn);
    zero_acc(dGc);
    auto qraw = [&](int r, int c) -> float {
        return r < ci.len ? bf2f(p.q[((ci.t0 + r) * p.Hk + hq) * D + c]) : 0.f;
    };
    auto kraw = [&](int r, int c) -> float {
        return bf2f(*reinterpret_cast<const __nv_bfloat16*>(sK.ptr(r, c)));
    };
#define FRAG_LOOP(NT_)                                                                          \
    _Pragma("unroll") for (int nt = 0; nt < NT_; ++nt) _Pragma("unroll") for (int e = 0; e < 4; ++e)
#define FRAG_RC(M0_, N0_)                                                                       \
    const int r = (M0_) + frag_g() + 8 * (e >> 1);                                              \
    const int c = (N0_) + nt * 8 + 2 * frag_c() + (e & 1)

    // ---- forward recompute ------------------------------------------------
    // kd' -> X1, ki' -> X2 ; A = strict_lower(beta kd' ki'^T)
    build_tile<F_KDP, D, KDA, false>(sX1, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f);
    build_tile<F_KIP, D, KDA, false>(sX2, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f);
    __syncthreads();
    {
        float acc[1][4][4];
        zero_acc(acc);
        warp_mma<1, 4, A_ROW, B_COL>(acc, sX1, sX2, mC, nC, 0, D);
        frag_foreach(acc, mC, nC, [&](int r, int c, float a0, float a1) {
            *reinterpret_cast<uint32_t*>(sA.ptr(r, c)) =
                pack_bf16(c < r ? sBeta[r] * a0 : 0.f, c + 1 < r ? sBeta[r] * a1 : 0.f);
        });
    }
    __syncthreads();
    // qd' -> X1 ; P = lower(qd' ki'^T)
    build_tile<F_KDP, D, KDA, true>(sX1, sX1, p.q, p, ci, hq, G, sInvQ, nullptr, p.scale,
                                    static_cast<const decltype(sX1)*>(nullptr), p.Hk);
    __syncthreads();
    {
        float acc[1][4][4];
        zero_acc(acc);
        warp_mma<1, 4, A_ROW, B_COL>(acc, sX1, sX2, mC, nC, 0, D);
        frag_foreach(acc, mC, nC, [&](int r, int c, float a0, float a1) {
            *reinterpret_cast<uint32_t*>(sP.ptr(r, c)) = pack_bf16(c <= r ? a0 : 0.f, c + 1 <= r ? a1 : 0.f);
        });
    }
    __syncthreads();
    // kd -> X1 ; X = kd S0 ; beta (V - X) -> V (hi) and U (lo) ; dqd = dO S0^T
    build_tile<F_KD, D, KDA, false>(sX1, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f);
    __syncthreads();
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_COL>(acc, sX1, sS0, mD, nD, 0, D);
        frag_foreach(acc, mD, nD, [&](int r, int c, float a0, float a1) {
            const float2 v = unpack_bf16(*reinterpret_cast<const uint32_t*>(sV.ptr(r, c)));
            store_pair(sV, PREC ? &sU : nullptr, r, c, sBeta[r] * (v.x - a0), sBeta[r] * (v.y - a1));
        });
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sDO, sS0, mD, nD, 0, D);
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float t = p.scale * acc[0][nt][e] * fac(F_KD, r, c);
            dQn[0][nt][e] += t;
            dGc[0][nt][e] += qraw(r, c) * sInvQ[r] * t;
        }
    }
    __syncthreads();
    // kr -> X1 ; du = P^T dO + kr dS_C -> X2
    build_tile<F_KR, D, KDA, false>(sX1, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f);
    __syncthreads();
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_COL, B_ROW>(acc, sP, sDO, mD, nD, 0, CH);
        warp_mma<1, NTD, A_ROW, B_COL>(acc, sX1, sDS, mD, nD, 0, D);
        frag_foreach(acc, mD, nD, [&](int r, int c, float a0, float a1) {
            *reinterpret_cast<uint32_t*>(sX2.ptr(r, c)) = pack_bf16(a0, a1);
        });
    }
    __syncthreads();
    // dY = T^T du ; dv = beta dY ; dbeta += <dY, beta E> ; dY -> X2
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_COL, B_ROW>(acc, sT, sX2, mD, nD, 0, CH);
        float rs[2] = {0.f, 0.f};
        frag_foreach(acc, mD, nD, [&](int r, int c, float a0, float a1) {
            float2 be = unpack_bf16(*reinterpret_cast<const uint32_t*>(sV.ptr(r, c)));
            if (PREC) {
                const float2 bl = unpack_bf16(*reinterpret_cast<const uint32_t*>(sU.ptr(r, c)));
                be.x += bl.x;
                be.y += bl.y;
            }
            rs[(r - mD) >> 3] += a0 * be.x + a1 * be.y;
            if (r < ci.len)
                *reinterpret_cast<uint32_t*>(p.dv + ((ci.t0 + r) * p.H + h) * D + c) =
                    pack_bf16(sBeta[r] * a0, sBeta[r] * a1);
        });
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
            rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
        }
        if (frag_c() == 0) {
            sDb[(warp >> 2) * CH + mD + frag_g()] = rs[0];
            sDb[(warp >> 2) * CH + mD + frag_g() + 8] = rs[1];
        }
        __syncthreads();
        frag_foreach(acc, mD, nD, [&](int r, int c, float a0, float a1) {
            *reinterpret_cast<uint32_t*>(sX2.ptr(r, c)) = pack_bf16(a0, a1);
        });
    }
    __syncthreads();
    // dkd (from E) = -beta (dY S0^T) ; u = T (beta E) -> U (hi) and V (lo)
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sX2, sS0, mD, nD, 0, D);
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float t = -sBeta[r] * acc[0][nt][e] * fac(F_KD, r, c);
            dKn[0][nt][e] += t;
            dGc[0][nt][e] += kraw(r, c) * sInvK[r] * t;
        }
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sT, sV, mD, nD, 0, CH);
        if (PREC) warp_mma<1, NTD, A_ROW, B_ROW>(acc, sT, sU, mD, nD, 0, CH);
        __syncthreads();
        frag_foreach(acc, mD, nD, [&](int r, int c, float a0, float a1) {
            store_pair(sU, PREC ? &sV : nullptr, r, c, a0, a1);
        });
    }
    __syncthreads();

    // ---- reverse pass, state-free part -----------------------------------
    // dkr = u dS_C^T ; dgT (kr part) = colsum(dkr . kr)
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sU, sDS, mD, nD, 0, D);
        if (PREC) warp_mma<1, NTD, A_ROW, B_ROW>(acc, sV, sDS, mD, nD, 0, D);
        float colsum[NTD][2];
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt) colsum[nt][0] = colsum[nt][1] = 0.f;
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float t = acc[0][nt][e] * fac(F_KR, r, c);  // dkr e^{gT-gc}
            dKn[0][nt][e] += t;
            const float kt = kraw(r, c) * sInvK[r] * t;
            dGc[0][nt][e] -= kt;
            colsum[nt][e & 1] += kt;
        }
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = colsum[nt][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (frag_g() == 0) sDgTp[(warp & 3) * D + nD + nt * 8 + 2 * frag_c() + j] = v;
            }
    }
    // dP = lower(dO u^T) -> P (hi) and the S0 space (lo)
    {
        float acc[1][4][4];
        zero_acc(acc);
        warp_mma<1, 4, A_ROW, B_COL>(acc, sDO, sU, mC, nC, 0, D);
        if (PREC) warp_mma<1, 4, A_ROW, B_COL>(acc, sDO, sV, mC, nC, 0, D);
        __syncthreads();  // every reader of P (du), S0 (Z) and dS_C (dkr) is done
        frag_foreach(acc, mC, nC, [&](int r, int c, float a0, float a1) {
            store_pair(sP, PREC ? &sDPlo : nullptr, r, c, c <= r ? a0 : 0.f, c + 1 <= r ? a1 : 0.f);
        });
    }
    // dA = -strict_lower(dY u^T) ; dbeta += rowsum(dA . A) ; A <- beta dA (hi, lo)
    {
        float acc[1][4][4];
        zero_acc(acc);
        warp_mma<1, 4, A_ROW, B_COL>(acc, sX2, sU, mC, nC, 0, D);
        if (PREC) warp_mma<1, 4, A_ROW, B_COL>(acc, sX2, sV, mC, nC, 0, D);
        float rs[2] = {0.f, 0.f};
        frag_foreach(acc, mC, nC, [&](int r, int c, float a0, float a1) {
            const float2 av = unpack_bf16(*reinterpret_cast<const uint32_t*>(sA.ptr(r, c)));
            const float d0 = c < r ? -a0 : 0.f, d1 = c + 1 < r ? -a1 : 0.f;
            rs[(r - mC) >> 3] += d0 * av.x + d1 * av.y;
            store_pair(sA, PREC ? &sBDAlo : nullptr, r, c, sBeta[r] * d0, sBeta[r] * d1);
        });
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
            rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
        }
        if (frag_c() == 0) {
            sDb[(2 + (warp >> 2)) * CH + mC + frag_g()] = rs[0];
            sDb[(2 + (warp >> 2)) * CH + mC + frag_g() + 8] = rs[1];
        }
    }
    // ki' -> X1 (+ lo)
    build_tile<F_KIP, D, KDA, false>(sX1, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f, PREC ? &sKIlo : nullptr);
    __syncthreads();
    // dqd' = dP ki' ; dkd' = (beta dA) ki'
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sP, sX1, mD, nD, 0, CH);
        if (PREC) {
            warp_mma<1, NTD, A_ROW, B_ROW>(acc, sDPlo, sX1, mD, nD, 0, CH);
            warp_mma<1, NTD, A_ROW, B_ROW>(acc, sP, sKIlo, mD, nD, 0, CH);
        }
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float f = fac(F_KDP, r, c);
            dQn[0][nt][e] += p.scale * acc[0][nt][e] * f;
            dGc[0][nt][e] += tile_val(qraw(r, c), derived_m(sInvQ[r], p.scale, 1.f), f) * acc[0][nt][e];
        }
        zero_acc(acc);
        warp_mma<1, NTD, A_ROW, B_ROW>(acc, sA, sX1, mD, nD, 0, CH);
        if (PREC) {
            warp_mma<1, NTD, A_ROW, B_ROW>(acc, sBDAlo, sX1, mD, nD, 0, CH);
            warp_mma<1, NTD, A_ROW, B_ROW>(acc, sA, sKIlo, mD, nD, 0, CH);
        }
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float f = fac(F_KDP, r, c);
            dKn[0][nt][e] += acc[0][nt][e] * f;
            dGc[0][nt][e] += tile_val(kraw(r, c), derived_m(sInvK[r], 1.f, 1.f), f) * acc[0][nt][e];
        }
    }
    __syncthreads();
    // qd' -> X1, kd' -> X2 (+ lo) ; dki' = dP^T qd' + (beta dA)^T kd'
    build_tile<F_KDP, D, KDA, true>(sX1, sX1, p.q, p, ci, hq, G, sInvQ, nullptr, p.scale, PREC ? &sQDlo : nullptr,
                                    p.Hk);
    build_tile<F_KDP, D, KDA, false>(sX2, sK, nullptr, p, ci, h, G, sInvK, nullptr, 1.f, PREC ? &sKDlo : nullptr);
    __syncthreads();
    {
        float acc[1][NTD][4];
        zero_acc(acc);
        warp_mma<1, NTD, A_COL, B_ROW>(acc, sP, sX1, mD, nD, 0, CH);
        warp_mma<1, NTD, A_COL, B_ROW>(acc, sA, sX2, mD, nD, 0, CH);
        if (PREC) {
            warp_mma<1, NTD, A_COL, B_ROW>(acc, sDPlo, sX1, mD, nD, 0, CH);
            warp_mma<1, NTD, A_COL, B_ROW>(acc, sP, sQDlo, mD, nD, 0, CH);
            warp_mma<1, NTD, A_COL, B_ROW>(acc, sBDAlo, sX2, mD, nD, 0, CH);
            warp_mma<1, NTD, A_COL, B_ROW>(acc, sA, sKDlo, mD, nD, 0, CH);
        }
        FRAG_LOOP(NTD) {
            FRAG_RC(mD, nD);
            const float f = fac(F_KIP, r, c);
            dKn[0][nt][e] += acc[0][nt][e] * f;
            dGc[0][nt][e] -= tile_val(kraw(r, c), derived_m(sInvK[r], 1.f, 1.f), f) * acc[0][nt][e];
        }
    }
#undef FRAG_LOOP
#undef FRAG_RC

    // ---- epilogue -----------------------------------------------------------
    // row dots <dqn, qn>, <dkn, kn>
    float qn[NTD][4], kn[NTD][4];
    {
        float rq[2] = {0.f, 0.f}, rk[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = mD + frag_g() + 8 * hf, c = nD + nt * 8 + 2 * frag_c();
                float2 qv = make_float2(0.f, 0.f);
                if (r < ci.len)
                    qv = unpack_bf16(*reinterpret_cast<const uint32_t*>(p.q + ((ci.t0 + r) * p.Hk + hq) * D + c));
                const float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t*>(sK.ptr(r, c)));
                qn[nt][2 * hf] = qv.x * sInvQ[r];
                qn[nt][2 * hf + 1] = qv.y * sInvQ[r];
                kn[nt][2 * hf] = kv.x * sInvK[r];
                kn[nt][2 * hf + 1] = kv.y * sInvK[r];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int e = 2 * hf + j;
                    rq[hf] += dQn[0][nt][e] * qn[nt][e];
                    rk[hf] += dKn[0][nt][e] * kn[nt][e];
                }
            }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            rq[i] += __shfl_xor_sync(0xffffffffu, rq[i], 1);
            rq[i] += __shfl_xor_sync(0xffffffffu, rq[i], 2);
            rk[i] += __shfl_xor_sync(0xffffffffu, rk[i], 1);
            rk[i] += __shfl_xor_sync(0xffffffffu, rk[i], 2);
        }
        if (frag_c() == 0) {
            const int half = warp >> 2;
            sRowQ[half * CH + mD + frag_g()] = rq[0];
            sRowQ[half * CH + mD + frag_g() + 8] = rq[1];
            sRowK[half * CH + mD + frag_g()] = rk[0];
            sRowK[half * CH + mD + frag_g() + 8] = rk[1];
        }
    }
    __syncthreads();
    // dq, dk stores; dgc -> fp32 scratch over the state tiles (their last
    // readers, the residual tiles of the precise mode, are behind the barrier above)
    float* sDgc = reinterpret_cast<float*>(smem + SM::oS0);  // [C][D]
#pragma unroll
    for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = mD + frag_g() + 8 * hf, c = nD + nt * 8 + 2 * frag_c();
            const float tq = sRowQ[r] + sRowQ[CH + r], tk = sRowK[r] + sRowK[CH + r];
            float oq[2], ok[2], og[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int e = 2 * hf + j;
                oq[j] = (dQn[0][nt][e] - qn[nt][e] * tq) * sInvQ[r];
                ok[j] = (dKn[0][nt][e] - kn[nt][e] * tk) * sInvK[r];
                og[j] = dGc[0][nt][e];
            }
            if (r < ci.len) {
                const size_t o = ((ci.t0 + r) * p.H + h) * D + c;
                *reinterpret_cast<uint32_t*>(p.dq + o) = pack_bf16(oq[0], oq[1]);
                *reinterpret_cast<uint32_t*>(p.dk + o) = pack_bf16(ok[0], ok[1]);
            }
            *reinterpret_cast<float2*>(sDgc + r * D + c) = make_float2(og[0], og[1]);
        }
    // dbeta in logit space
    for (int r = threadIdx.x; r < ci.len; r += blockDim.x) {
        const float db = ((sDb[r] + sDb[CH + r]) + sDb[2 * CH + r]) + sDb[3 * CH + r];
        p.dbeta[(ci.t0 + r) * p.H + h] = __float2bfloat16((1.f - sBeta[r]) * db);
    }
    auto dgT_of = [&](int d) -> float {
        return (((sDgTs[d] + sDgTp[d]) + sDgTp[D + d]) + sDgTp[2 * D + d]) + sDgTp[3 * D + d];
    };
    __syncthreads();

    // reverse cumsum of dgc plus the chunk constant dgT, then the gate front end
    if constexpr (!KDA) {
        // channel sums first (the scalar gate's gradient is the channel sum)
        for (int rr = 0; rr < CH / 8; ++rr) {  // warp w sums rows 8w .. 8w+7
            const int r = warp * (CH / 8) + rr;
            float s = 0.f;
            for (int d = lane; d < D; d += 32) s += sDgc[r * D + d];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) sMisc[r] = s;
        }
        __syncthreads();
        if (warp == 0) {
            float t = 0.f;
            for (int d = lane; d < D; d += 32) t += dgT_of(d);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            // suffix sums over 64 rows: lane holds rows 2*lane, 2*lane+1
            const float a = sMisc[2 * lane], b = sMisc[2 * lane + 1];
            float s = a + b, incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float v = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += v;
            }
            // incl = sum of rows >= 2*lane
            const float suf0 = incl + t, suf1 = incl - a + t;
            if (2 * lane < ci.len) p.dg[(ci.t0 + 2 * lane) * p.H + h] = suf0;
            if (2 * lane + 1 < ci.len) p.dg[(ci.t0 + 2 * lane + 1) * p.H + h] = suf1;
        }
    } else {
        // suffix sums per channel in place (one thread per channel), then the gate
        // chain elementwise over all threads with per-channel partial sums
        for (int d = threadIdx.x; d < D; d += blockDim.x) {
            float acc = dgT_of(d);
            for (int r = CH - 1; r >= 0; --r) {
                acc += sDgc[r * D + d];
                sDgc[r * D + d] = acc;
            }
        }
        __syncthreads();
        const float ea = expf(p.A_log[h]);
        constexpr int RSTEP = 256 / D;  // rows handled per pass (threads per channel)
        const int d = threadIdx.x % D, r0 = threadIdx.x / D;
        const float dt = p.dt_bias[h * D + d];
        float ddt = 0.f, dA_acc = 0.f;
        for (int r = r0; r < ci.len; r += RSTEP) {
            const size_t o = ((ci.t0 + r) * p.H + h) * D + d;
            const float x = bf2f(p.g_raw[o]) + dt;
            const float dgl = sDgc[r * D + d];
            float dA;
            const float draw = kda_gate_bwd(p.kda_gate, p.gate_scale, ea, x, dgl, dA);
            p.dg_raw[o] = __float2bfloat16(draw);
            ddt += draw;
            dA_acc += dA;
        }
        __syncthreads();  // sDgc reads done; reuse the row-sum scratch for the partials
        sRowQ[threadIdx.x] = ddt;  // [RSTEP][D] (256 floats: rowq and rowk are contiguous)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dA_acc += __shfl_xor_sync(0xffffffffu, dA_acc, o);
        if (lane == 0) sMisc[warp] = dA_acc;
        __syncthreads();
        if (threadIdx.x < D) {
            float t = 0.f;
            for (int j = 0; j < RSTEP; ++j) t += sRowQ[j * D + threadIdx.x];
            atomicAdd(&p.ddt_bias[h * D + threadIdx.x], t);
        }
        if (threadIdx.x == 0) {
            float t = 0.f;
            for (int w = 0; w < 8; ++w) t += sMisc[w];
            atomicAdd(&p.dA_log[h], t);
        }
    }
}

template <int D, bool KDA>
static cudaError_t launch_main_t(const Params& p, cudaStream_t s) {
    const int bytes = MainSmem<D, KDA>::bytes;
    cudaError_t e = cudaFuncSetAttribute(k_main<D, KDA>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_chunks, p.H);
    k_main<D, KDA><<<grid, 256, bytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_main(const Params& p, cudaStream_t s) {
    if (p.max_chunks == 0) return cudaSuccess;
    if (p.D == 128) return p.kda ? launch_main_kda(p, s) : launch_main_gdn(p, s);
    if (p.D == 128) return p.kda ? launch_main_t<128, true>(p, s) : launch_main_t<128, false>(p, s);
    return p.kda ? launch_main_t<64, true>(p, s) : launch_main_t<64, false>(p, s);
}

}  // namespace gdr
