// Chunk-parallel main backward on tcgen05 (GDN, D = 128): one CTA (16 warps)
// per (chunk, head).  Same algebra as the warp-level kernel in gdr_main.cu, with
// every product issued as a 128-row tcgen05 MMA into tensor memory.
//
// Products are written feature-major where the natural output is C x D: the
// accumulator holds X^T (lane = feature d or value channel j, column = token
// row r), so a thread owns one feature for 16 rows and the per-row gate
// factors are per-thread scalars.  C x C products stack two 64-row operands
// into one 128-row operand ([kd'; qd'] ki'^T gives A and P; [dO; dY] u^T gives
// dP and dA).  With S0 = chunk-start state, dS = state gradient at the chunk end (both
// saved value-major, [dv][dk], so the operand major-ness below reads them transposed):
//   G1  [A_raw; P]   = [kd'; qd'] ki'^T                 G7  Z^T    = S0 dY^T
//   G2  X^T          = S0^T kd^T                        G8  dkr^T  = dS u^T
//   G3  dqd^T        = S0 dO^T                          G9  [dP; dA] = [dO; dY] u^T
//   G4  u^T          = (beta E)^T T^T                   G10 [dqd', dkd']^T = ki'^T [dP; beta dA]^T
//   G5  du^T         = dO^T P + dS^T kr^T               G11 dki'^T = qd'^T dP + kd'^T (beta dA)
//   G6  dY^T         = du^T T
// followed by the elementwise assembly of "FlashKDA之backward（K1）" (§3.2-§3.3, §5).
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"

namespace gdr {

namespace {

constexpr int TC_D = 128;
// shared-memory map (bytes from the 1024-aligned base)
constexpr int oK = 0;             // k           [64][128]
constexpr int oV = 16384;         // v -> beta E [64][128]
constexpr int oDOY = 32768;       // [dO; dY]    [128][128]
constexpr int oS0 = 65536;        // S0 [128][128]; later kd' [64][128]; last, dgc fp32
constexpr int oDS = 98304;        // dS [128][128]; later [dP; beta dA] [128][64]
constexpr int oT = 131072;        // T  [64][64]
constexpr int oA = 139264;        // A  [64][64]
constexpr int oP = 147456;        // P  [64][64]
constexpr int oW0 = 155648;       // work: [kd'; qd'] (W0..W1), kd, ki'
constexpr int oW1 = 172032;       // work: u
constexpr int oW2 = 188416;       // work: ki', kr -> du, qd'
constexpr int oSmall = 204800;
// small arrays (floats)
constexpr int NCOL = 16;  // columns per thread (16 warps: 4 lane quarters x 4 column quarters)
constexpr int nInvQ = 64, nInvK = 64, nBeta = 64, nFac = 256, nGate = 128, nDgTs = 128, nDgTp = 512,
              nDbP = 64, nDbA = 256, nRow = 256 * 3, nMisc = 64;
constexpr int SMALL_FLOATS = nInvQ + nInvK + nBeta + nFac + nGate + nDgTs + nDgTp + nDbP + nDbA + nRow + nMisc;
constexpr int SMEM_BYTES = oSmall + SMALL_FLOATS * 4 + 64 + 1024;  // + mbarrier/tmem slot + alignment
// tensor-memory columns
constexpr uint32_t R_A = 0, R_B = 128, R_C = 192, R_D = 256, R_Q = 320, R_K = 384;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// cp.async of the chunk rows of a token-major [T,H,D] tensor into a SW128 tile (rows >= len zero-filled)
__device__ __forceinline__ void load_rows_sw(unsigned char* tile, int rows, const __nv_bfloat16* src,
                                             const Params& p, const ChunkInfo& ci, int h) {
    for (int i = threadIdx.x; i < CH * (TC_D / 8); i += blockDim.x) {
        const int r = i / (TC_D / 8), j = i % (TC_D / 8);
        const bool ok = r < ci.len;
        cp_async16(tile + tc::sw_chunk(r, j, rows), src + ((ci.t0 + (ok ? r : 0)) * p.H + h) * TC_D + j * 8, ok);
    }
}
// cp.async of a contiguous row-major ROWS x COLS bf16 tile into a SW128 tile
template <int ROWS, int COLS>
__device__ __forceinline__ void load_tile_sw(unsigned char* tile, const __nv_bfloat16* src) {
    for (int i = threadIdx.x; i < ROWS * (COLS / 8); i += blockDim.x) {
        const int r = i / (COLS / 8), j = i % (COLS / 8);
        cp_async16(tile + tc::sw_chunk(r, j, ROWS), src + (size_t)r * COLS + j * 8, true);
    }
}

// dst rows row0.. of a SW128 tile with `rows` rows: bf16(x * m_r * e^{factor KIND}(r)),
// x from the k tile (smem) or from global q; per-row factors from the table.
template <bool SRC_GLOBAL>
__device__ __forceinline__ void build_sw(unsigned char* dst, int rows, int row0, const unsigned char* sK,
                                         const __nv_bfloat16* gq, const Params& p, const ChunkInfo& ci, int h,
                                         const float* fac, const float* inv, float mul) {
    for (int i = threadIdx.x; i < CH * (TC_D / 8); i += blockDim.x) {
        const int r = i / (TC_D / 8), j = i % (TC_D / 8);
        uint4 v;
        if (SRC_GLOBAL) {
            v = r < ci.len ? *reinterpret_cast<const uint4*>(gq + ((ci.t0 + r) * p.H + h) * TC_D + j * 8)
                           : make_uint4(0, 0, 0, 0);
        } else {
            v = *reinterpret_cast<const uint4*>(sK + tc::sw_chunk(r, j, 64));
        }
        const float m = derived_m(inv[r], mul, 1.f), f = fac[r];
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = unpack_bf16(w[e]);
            w[e] = pack_bf16(x.x * m * f, x.y * m * f);
        }
        *reinterpret_cast<uint4*>(dst + tc::sw_chunk(row0 + r, j, rows)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

__global__ void __launch_bounds__(512, 1) k_main_tc(const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int chunk = blockIdx.x, h = blockIdx.y;
    ChunkInfo ci;
    if (!lookup_chunk(chunk, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, ci)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hc = warp >> 2;  // TMEM lane quarter, column quarter
    const int L = 32 * q4 + lane;             // this thread's TMEM lane (a feature, or a stacked row)
    const int c0 = NCOL * hc;                 // first of this thread's 16 columns

    unsigned char *sK = smem + oK, *sV = smem + oV, *sDOY = smem + oDOY, *sS0 = smem + oS0, *sDS = smem + oDS,
                  *sT = smem + oT, *sA = smem + oA, *sP = smem + oP, *sW0 = smem + oW0, *sW1 = smem + oW1,
                  *sW2 = smem + oW2;
    float* fsm = reinterpret_cast<float*>(smem + oSmall);
    float* sInvQ = fsm;
    float* sInvK = sInvQ + nInvQ;
    float* sBeta = sInvK + nInvK;
    float* sFac = sBeta + nBeta;     // [4][64] e^{gc}, e^{gc-ref}, e^{ref-gc}, e^{gT-gc}
    float* sGate = sFac + nFac;      // gc[64], ref, gT
    float* sDgTs = sGate + nGate;    // [128] state part of dgT
    float* sDgTp = sDgTs + nDgTs;    // [4][128] kr part of dgT per column quarter
    float* sDbP = sDgTp + nDgTp;     // [64] <dY, beta E> per row
    float* sDbA = sDbP + nDbP;       // [4][64] rowsum(dA . A) per column quarter
    float* sRow = sDbA + nDbA;       // [3][4][64] row reductions
    float* sMisc = sRow + nRow;      // [64]
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sMisc + nMisc);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 1);
    const uint32_t mb = smem_u32(mbar);

    Gates<TC_D, false> G;
    G.gc = sGate;
    G.ref = sGate + CH;
    G.gT = sGate + CH + 1;

    const size_t tdd = ((size_t)chunk * p.H + h) * TC_D * TC_D;
    const size_t tcc = ((size_t)chunk * p.H + h) * CH * CH;

    // ---- set-up: tensor memory, mbarrier, loads ---------------------------------
    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) tc::mbar_init(mb, 1);
    load_rows_sw(sK, 64, p.k, p, ci, h);
    load_rows_sw(sV, 64, p.v, p, ci, h);
    load_rows_sw(sDOY, 128, p.dO, p, ci, h);
    load_tile_sw<TC_D, TC_D>(sS0, p.S0 + tdd);
    load_tile_sw<TC_D, TC_D>(sDS, p.dS + tdd);
    load_tile_sw<CH, CH>(sT, p.Tm + tcc);
    cp_async_commit();
    load_gates<TC_D, false>(p, ci, h, G, false);
    load_beta(p, ci, h, sBeta);
    row_inv_norms_global<TC_D>(p.q, p, ci, h, sInvQ);
    cp_async_wait<0>();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    uint32_t phase = 0;
    bool ok = true;
    auto sync_all = [&]() {  // make smem writes visible to the tensor cores and order TMEM use
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    // Waits for the last commit.  If the tensor cores do not answer within the
    // bounded spin, every thread learns it from the vote, the status word records
    // it, the tensor memory is released and the CTA returns.
    auto wait_mma = [&]() -> bool {
        ok = tc::mbar_wait(mb, phase);
        phase ^= 1;
        tc::fence_after();
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(p.status, ST_MMA_TIMEOUT);
            tc::fence_before();
            __syncthreads();
            if (warp == 0) tc::dealloc(tmem, 512);
            return false;
        }
        return true;
    };
    auto tl = [&](uint32_t col) { return tmem + ((uint32_t)(32 * q4) << 16) + col; };

    // k norms (4 threads per row), gate factor table, dgT state part
    {
        const int r = tid >> 2, part = tid & 3;
        float s = 0.f;
        if (r < CH) {
            for (int j = part * 4; j < part * 4 + 4; ++j) {
                uint4 v = *reinterpret_cast<const uint4*>(sK + tc::sw_chunk(r, j, 64));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack_bf16(w[e]);
                    s += f.x * f.x + f.y * f.y;
                }
            }
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (r < CH && part == 0) sInvK[r] = rsqrtf(s + 1e-6f);
    }
    for (int r = tid; r < CH; r += blockDim.x) {
        sFac[0 * CH + r] = gate_factor<F_KD>(G, r, 0);
        sFac[1 * CH + r] = gate_factor<F_KDP>(G, r, 0);
        sFac[2 * CH + r] = gate_factor<F_KIP>(G, r, 0);
        sFac[3 * CH + r] = gate_factor<F_KR>(G, r, 0);
    }
    {  // e^{gT} rowsum(dS . S0) per key channel: a column sum of the value-major tiles
        const int cp = tid >> 3, g = tid & 7;  // column pair, row group
        float s0 = 0.f, s1 = 0.f;
        for (int j = g; j < TC_D; j += 8) {
            const float2 a = unpack_bf16(*reinterpret_cast<const uint32_t*>(sS0 + tc::sw_off(j, 2 * cp, 128)));
            const float2 b = unpack_bf16(*reinterpret_cast<const uint32_t*>(sDS + tc::sw_off(j, 2 * cp, 128)));
            s0 += a.x * b.x;
            s1 += a.y * b.y;
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (g == 0) {
            const float eg = __expf(G.gTv(0));
            sDgTs[2 * cp] = s0 * eg;
            sDgTs[2 * cp + 1] = s1 * eg;
        }
    }
    __syncthreads();
    const float* facKD = sFac;
    const float* facKDP = sFac + CH;
    const float* facKIP = sFac + 2 * CH;
    const float* facKR = sFac + 3 * CH;

    // per-thread accumulators (feature L, rows c0 .. c0+15)
    float dQn[NCOL], dKn[NCOL], dGc[NCOL], v[NCOL], qk[NCOL];
#pragma unroll
    for (int i = 0; i < NCOL; ++i) dQn[i] = dKn[i] = dGc[i] = 0.f;
    // byte offset of element (row c0 + i, column L) in a token-major SW128 tile with `rows` rows;
    // c0 is a multiple of 16, so (row & 7) == (i & 7) is known at compile time
    const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
    auto tok = [&](int rows, int i) -> uint32_t {
        return (uint32_t)((L >> 6) * rows * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
    };
    auto tok_bf = [&](const unsigned char* base, int rows, int i) -> float {
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + tok(rows, i)));
    };
    // raw q and k of this thread's feature and rows, staged once in tensor memory
    {
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {
            const int r = c0 + i;
            qk[i] = r < ci.len ? bf2f(p.q[((ci.t0 + r) * p.H + h) * TC_D + L]) : 0.f;
        }
        tc::st16(tl(R_Q + c0), qk);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) qk[i] = tok_bf(sK, 64, i);
        tc::st16(tl(R_K + c0), qk);
    }

    // ---- G1: [A_raw; P] = [kd'; qd'] ki'^T ----------------------------------------
    build_sw<false>(sW0, 128, 0, sK, nullptr, p, ci, h, facKDP, sInvK, 1.f);        // kd'
    build_sw<true>(sW0, 128, 64, sK, p.q, p, ci, h, facKDP, sInvQ, p.scale);         // qd'
    build_sw<false>(sW2, 64, 0, sK, nullptr, p, ci, h, facKIP, sInvK, 1.f);         // ki'
    sync_all();
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 0, 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_B, tc::kdesc(sb + oW0, 128, 0, k), tc::kdesc(sb + oW2, 64, 0, k), id, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_B + c0), v);
    {
        const bool isA = L < 64;
        const int r = isA ? L : L - 64;
        unsigned char* dst = isA ? sA : sP;
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s0 = c0 + jc * 8 + 2 * e;
                float a0 = v[jc * 8 + 2 * e], a1 = v[jc * 8 + 2 * e + 1];
                if (isA) {
                    a0 = s0 < r ? sBeta[r] * a0 : 0.f;
                    a1 = s0 + 1 < r ? sBeta[r] * a1 : 0.f;
                } else {
                    a0 = s0 <= r ? a0 : 0.f;
                    a1 = s0 + 1 <= r ? a1 : 0.f;
                }
                w[e] = pack_bf16(a0, a1);
            }
            *reinterpret_cast<uint4*>(dst + tc::sw_chunk(r, (c0 >> 3) + jc, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    __syncthreads();  // everyone is past G1's wait: its operands may be overwritten
    build_sw<false>(sW0, 64, 0, sK, nullptr, p, ci, h, facKD, sInvK, 1.f);   // kd
    sync_all();

    // ---- G2: X^T = S0^T kd^T ; G3: dqd^T = S0 dO^T -----------------------------------
    if (tid == 0) {
        constexpr uint32_t id2 = tc::idesc(128, 64, 0, 0), id3 = tc::idesc(128, 64, 1, 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_C, tc::kdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oW0, 64, 0, k), id2, k > 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_D, tc::mdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oDOY, 128, 0, k), id3, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_C + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // beta E = beta (V - X), in place of V (lane = value channel)
        const int r = c0 + i;
        __nv_bfloat16* pv = reinterpret_cast<__nv_bfloat16*>(sV + tok(64, i));
        *pv = __float2bfloat16(sBeta[r] * (__bfloat162float(*pv) - v[i]));
    }
    tc::ld16(tl(R_D + c0), v);
    tc::ld16(tl(R_Q + c0), qk);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // dqd (lane = key channel)
        const int r = c0 + i;
        const float t = p.scale * v[i] * facKD[r];
        dQn[i] += t;
        dGc[i] += qk[i] * sInvQ[r] * t;
    }
    build_sw<false>(sW2, 64, 0, sK, nullptr, p, ci, h, facKR, sInvK, 1.f);   // kr (ki' is dead)
    sync_all();

    // ---- G4: u^T = (beta E)^T T^T ; G5: du^T = dO^T P + dS^T kr^T -----------------------
    if (tid == 0) {
        constexpr uint32_t id4 = tc::idesc(128, 64, 1, 0), id5a = tc::idesc(128, 64, 1, 1),
                           id5b = tc::idesc(128, 64, 0, 0);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oV, 64, 0, k), tc::kdesc(sb + oT, 64, 0, k), id4, k > 0);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_C, tc::mdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oP, 64, 0, k), id5a, k > 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_C, tc::kdesc(sb + oDS, 128, 0, k), tc::kdesc(sb + oW2, 64, 0, k), id5b, 1);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    // u^T and du^T are stored feature-major ([j][r], 128 rows x 64 columns): 16-byte row stores
    auto store_fm = [&](unsigned char* dst) {
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = pack_bf16(v[jc * 8 + 2 * e], v[jc * 8 + 2 * e + 1]);
            *reinterpret_cast<uint4*>(dst + tc::sw_chunk(L, (c0 >> 3) + jc, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    };
    tc::ld16(tl(R_B + c0), v);
    store_fm(sW1);  // u^T
    tc::ld16(tl(R_C + c0), v);
    store_fm(sW2);  // du^T over kr
    sync_all();

    // ---- G6: dY^T = du^T T ------------------------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id6 = tc::idesc(128, 64, 0, 1);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oW2, 128, 0, k), tc::mdesc(sb + oT, 64, 0, k), id6, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_D + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {
        const int r = c0 + i;
        if (r < ci.len) p.dv[((ci.t0 + r) * p.H + h) * TC_D + L] = __float2bfloat16(sBeta[r] * v[i]);
        *reinterpret_cast<__nv_bfloat16*>(sDOY + tok(128, i) + 64 * 128) = __float2bfloat16(v[i]);  // dY below dO
    }
    sync_all();

    // ---- G7: Z^T = S0 dY^T ; G8: dkr^T = dS u^T ; G9: [dP; dA]_raw = [dO; dY] u^T ------------
    if (tid == 0) {
        constexpr uint32_t id7 = tc::idesc(128, 64, 1, 0), id8 = tc::idesc(128, 64, 1, 1),
                           id9 = tc::idesc(128, 64, 0, 1);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oDOY, 128, 64, k), id7, k > 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_C, tc::mdesc(sb + oDS, 128, 0, k), tc::mdesc(sb + oW1, 128, 0, k), id8, k > 0);
        for (int k = 0; k < TC_D; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oW1, 128, 0, k), id9, k > 0);
        tc::commit(mb);
    }
    // while the tensor cores run: <dY, beta E> per row (token-major, 4 threads per row)
    if (tid < 4 * CH) {
        const int r = tid >> 2, part = tid & 3;
        float s2 = 0.f;
        for (int j = part * 4; j < part * 4 + 4; ++j) {
            uint4 a = *reinterpret_cast<const uint4*>(sDOY + tc::sw_chunk(64 + r, j, 128));
            uint4 b = *reinterpret_cast<const uint4*>(sV + tc::sw_chunk(r, j, 64));
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = unpack_bf16(wa[e]), fb = unpack_bf16(wb[e]);
                s2 += fa.x * fb.x + fa.y * fb.y;
            }
        }
        s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
        s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
        if (part == 0) sDbP[r] = s2;
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_K + c0), qk);  // raw k
    tc::ld16(tl(R_B + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // dkd (from E) = -beta Z
        const int r = c0 + i;
        const float t = -sBeta[r] * v[i] * facKD[r];
        dKn[i] += t;
        dGc[i] += qk[i] * sInvK[r] * t;
    }
    tc::ld16(tl(R_C + c0), v);
    {
        float dgt = 0.f;
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dkr
            const int r = c0 + i;
            const float t = v[i] * facKR[r];
            dKn[i] += t;
            const float kt = qk[i] * sInvK[r] * t;
            dGc[i] -= kt;
            dgt += kt;
        }
        sDgTp[hc * TC_D + L] = dgt;
    }
    tc::ld16(tl(R_D + c0), v);
    {
        // lanes 0..63: dP rows, lanes 64..127: dA rows ; [dP; beta dA] -> dS space [128][64]
        const bool isP = L < 64;
        const int r = isP ? L : L - 64;
        float dbs = 0.f;
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            uint32_t w[4];
            const uint4 av = *reinterpret_cast<const uint4*>(sA + tc::sw_chunk(r, (c0 >> 3) + jc, 64));
            const uint32_t wa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s0 = c0 + jc * 8 + 2 * e;
                float a0 = v[jc * 8 + 2 * e], a1 = v[jc * 8 + 2 * e + 1];
                if (isP) {
                    a0 = s0 <= r ? a0 : 0.f;
                    a1 = s0 + 1 <= r ? a1 : 0.f;
                } else {
                    a0 = s0 < r ? -a0 : 0.f;
                    a1 = s0 + 1 < r ? -a1 : 0.f;
                    const float2 aa = unpack_bf16(wa[e]);
                    dbs += a0 * aa.x + a1 * aa.y;
                    a0 *= sBeta[r];
                    a1 *= sBeta[r];
                }
                w[e] = pack_bf16(a0, a1);
            }
            *reinterpret_cast<uint4*>(sDS + tc::sw_chunk(L, (c0 >> 3) + jc, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (!isP) sDbA[hc * CH + r] = dbs;
    }
    __syncthreads();  // dS, S0, kd and du are dead
    build_sw<false>(sW0, 64, 0, sK, nullptr, p, ci, h, facKIP, sInvK, 1.f);        // ki'
    build_sw<true>(sW2, 64, 0, sK, p.q, p, ci, h, facKDP, sInvQ, p.scale);          // qd'
    build_sw<false>(sS0, 64, 0, sK, nullptr, p, ci, h, facKDP, sInvK, 1.f);         // kd'
    sync_all();

    // ---- G10: [dqd', dkd']^T = ki'^T [dP; beta dA]^T ; G11: dki'^T = qd'^T dP + kd'^T (beta dA) --
    if (tid == 0) {
        constexpr uint32_t id10 = tc::idesc(128, 128, 1, 0), id11 = tc::idesc(128, 64, 1, 1);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_A, tc::mdesc(sb + oW0, 64, 0, k), tc::kdesc(sb + oDS, 128, 0, k), id10, k > 0);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oW2, 64, 0, k), tc::mdesc(sb + oDS, 128, 0, k), id11, k > 0);
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oS0, 64, 0, k), tc::mdesc(sb + oDS, 128, 64, k), id11, 1);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_Q + c0), qk);  // raw q
    tc::ld16(tl(R_A + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // dqd'
        const int r = c0 + i;
        const float f = facKDP[r];
        dQn[i] += p.scale * v[i] * f;
        dGc[i] += derived_val(qk[i], derived_m(sInvQ[r], p.scale, 1.f), f) * v[i];
    }
    tc::ld16(tl(R_K + c0), qk);  // raw k
    tc::ld16(tl(R_A + 64 + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // dkd'
        const int r = c0 + i;
        const float f = facKDP[r];
        dKn[i] += v[i] * f;
        dGc[i] += derived_val(qk[i], derived_m(sInvK[r], 1.f, 1.f), f) * v[i];
    }
    tc::ld16(tl(R_B + c0), v);
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {  // dki'
        const int r = c0 + i;
        const float f = facKIP[r];
        dKn[i] += v[i] * f;
        dGc[i] -= derived_val(qk[i], derived_m(sInvK[r], 1.f, 1.f), f) * v[i];
    }

    // ---- epilogue: L2 backward, dq / dk, dbeta, dg ---------------------------------------
    float* sRowQ = sRow;            // [4][64]
    float* sRowK = sRow + 256;      // [4][64]
    float* sRowG = sRow + 512;      // [4][64]
    tc::ld16(tl(R_Q + c0), v);      // raw q (k is in qk)
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {
        const int r = c0 + i;
        const float a = warp_sum(dQn[i] * v[i] * sInvQ[r]);
        const float b = warp_sum(dKn[i] * qk[i] * sInvK[r]);
        const float g = warp_sum(dGc[i]);
        if (lane == 0) {
            sRowQ[q4 * CH + r] = a;
            sRowK[q4 * CH + r] = b;
            sRowG[q4 * CH + r] = g;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NCOL; ++i) {
        const int r = c0 + i;
        if (r < ci.len) {
            const float tq = ((sRowQ[r] + sRowQ[CH + r]) + sRowQ[2 * CH + r]) + sRowQ[3 * CH + r];
            const float tk = ((sRowK[r] + sRowK[CH + r]) + sRowK[2 * CH + r]) + sRowK[3 * CH + r];
            const float qn = v[i] * sInvQ[r];
            const float kn = qk[i] * sInvK[r];
            const size_t o = ((ci.t0 + r) * p.H + h) * TC_D + L;
            p.dq[o] = __float2bfloat16((dQn[i] - qn * tq) * sInvQ[r]);
            p.dk[o] = __float2bfloat16((dKn[i] - kn * tk) * sInvK[r]);
        }
    }
    // dbeta (logit space)
    for (int r = tid; r < ci.len; r += blockDim.x) {
        const float dA_A = ((sDbA[r] + sDbA[CH + r]) + sDbA[2 * CH + r]) + sDbA[3 * CH + r];
        p.dbeta[(ci.t0 + r) * p.H + h] = __float2bfloat16((1.f - sBeta[r]) * (sDbP[r] + dA_A));
    }
    // dg: channel sums of dgc (per row), suffix sums over the rows, plus the chunk constant dgT
    if (warp == 0) {
        float t = 0.f;
        for (int d = lane; d < TC_D; d += 32)
            t += (((sDgTs[d] + sDgTp[d]) + sDgTp[TC_D + d]) + sDgTp[2 * TC_D + d]) + sDgTp[3 * TC_D + d];
        t = warp_sum(t);
        const int r0 = 2 * lane;
        const float a = ((sRowG[r0] + sRowG[CH + r0]) + sRowG[2 * CH + r0]) + sRowG[3 * CH + r0];
        const float b = ((sRowG[r0 + 1] + sRowG[CH + r0 + 1]) + sRowG[2 * CH + r0 + 1]) + sRowG[3 * CH + r0 + 1];
        float incl = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
        }
        if (r0 < ci.len) p.dg[(ci.t0 + r0) * p.H + h] = incl + t;
        if (r0 + 1 < ci.len) p.dg[(ci.t0 + r0 + 1) * p.H + h] = incl - a + t;
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_main_tc(const Params& p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(k_main_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.max_chunks, p.H);
    k_main_tc<<<grid, 512, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace gdr
