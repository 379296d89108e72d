// Chunk-parallel main backward on tcgen05 for D = 128 with the scalar (GDN) gate:
// persistent CTAs of 16 warps, one per SM, each looping over (chunk, head) items, the
// next item's operand tiles arriving by TMA while the current item's epilogue runs.
//
// With one log gate per token, every gated tile of the chunk algebra is a row scaling
// of the raw q or k tile: kd' = diag(invk e^{gc-ref}) k, qd' = diag(scale invq
// e^{gc-ref}) q, ki' = diag(invk e^{ref-gc}) k, kd = diag(invk e^{gc}) k,
// kr = diag(invk e^{gT-gc}) k.  So the tensor cores read the raw bf16 q and k tiles as
// they arrive (no derived tile is built) and the row factors are applied in fp32 where
// a product's result is read or where the next operand is written:
//   B1  G1  [A; P]_raw = [k; q] k^T       G2  X^T_raw = S0^T k^T    G5b du^T_raw = dS^T k^T
//   B2  G4  u^T  = (beta E)^T T^T         G5a du^T = dO^T P      (+ G5b x invk e^{gT-gc})
//   B3  G6  dY^T = du^T T
//   B4  G3/G7 [dqd^T, Z^T] = S0 [dO; dY]^T   G8 dkr^T = dS u^T   G9 [dP; dA]_raw = [dO; dY] u^T
//   B5  G10 [dqd', dkd']^T = k^T X10^T    G11 dki'^T = q^T X11_P + k^T X11_A
// A tcgen05.mma takes tens of cycles to issue whatever its size, so the groups of a batch
// are issued by lane 0 of different warps (one per SM sub-partition), each committing to
// the batch's barrier, and G3 waits for dY to run as one N = 128 product with G7.
// dv, dq and dk are staged token-major in shared tiles that are dead by then (du^T, u^T,
// A and P) and written by TMA stores; a chunk cut by its sequence's end copies its valid
// rows from the staged tile instead.
// with X10 = [dP; beta dA] scaled by the column factor invk_s e^{ref-gc_s} (ki' folded
// in) and X11 = [dP; beta dA] scaled by the row factors of qd' and kd'.  B1 needs no
// per-item preparation, so it is issued as soon as the tiles land and runs under the
// prologue (norms, gate factors, the state part of dgT).
//
// The gate gradient inside the chunk is taken in pair form ("FlashKDA之backward（K1）",
// §3.2(b), stable dgc): P[r][s] and A[r][s] depend on gc_r - gc_s, so each element adds
// t = dP P (or dA A) to row r and subtracts the same t from row s.  Both sides use one
// number, the bf16 element the products consumed, so the pairs cancel exactly in the
// reverse cumsum.  The other gate terms (qd through S0, kd through X, kr and gT) are
// summed per element over the channels as in the per-channel kernel.
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"

namespace gdr {

namespace {

constexpr int MD = 128;
constexpr int TILE = CH * MD * 2;  // 16 KB
// shared-memory map (bytes from the 1024-aligned base); later tenants after the arrows
constexpr int oKQ = 0;          // [k; q] token-major, 128 rows (k rows 0..63, q rows 64..127)
constexpr int oV = 32768;       // v -> beta E (token-major)
constexpr int oDOY = 49152;     // [dO; dY] token-major, 128 rows
constexpr int oS0 = 81920;      // S0 [j][d]
constexpr int oDS = 114688;     // dS [j][d] -> X10 [m][s] (+ X11 [m][s] at +16 KB)
constexpr int oT = 147456;      // T [r][s]
constexpr int oA = 155648;      // A = beta A_raw, strict lower [r][s]
constexpr int oP = 163840;      // P, lower [r][s]
constexpr int oU = 172032;      // u^T [j][r]
constexpr int oDU = 188416;     // du^T [j][r]
constexpr int oSmall = 204800;
constexpr int NCOL = 16;  // rows per thread (16 warps: 4 lane quarters x 4 row quarters)
// small arrays (floats)
constexpr int nInvQ = 64, nInvK = 64, nBeta = 128, nFac = 4 * 64, nTab = 6 * 64, nGate = 66, nPad = 62,
              nDgTs = 128, nDgTp = 512, nDbP = 64, nPairR = 512, nPairC = 256, nRowG = 256, nRow = 512, nTot = 128;
constexpr int SMALL_FLOATS = nInvQ + nInvK + nBeta + nFac + nTab + nGate + nPad + nDgTs + nDgTp + nDbP + nPairR +
                             nPairC + nRowG + nRow + nTot;
constexpr int SMEM_BYTES = oSmall + SMALL_FLOATS * 4 + 64 + 1024;  // + mbarriers / tmem slot + alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// tensor-memory columns
constexpr uint32_t R_A = 0, R_B = 128, R_C = 192, R_D = 256, R_Q = 320, R_K = 384, R_G5 = 448;
// combined row-factor tables (each [64])
enum Tab { T_CF = 0, T_KDF = 1, T_KRF = 2, T_RA = 3, T_RP = 4, T_RK = 5 };

struct GdnMaps {
    CUtensorMap q, k, v, dO, S0, dS, T, dq, dk, dv;
};
constexpr int STORE_TID = 96;  // the thread that issues the TMA stores of dq, dk and dv

}  // namespace

__global__ void __launch_bounds__(512, 1) k_main_gdn(const Params p, const __grid_constant__ GdnMaps m) {
    if (!states_header_ok(p)) {  // saved states of another variant or shape: write nothing
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, ST_STATES_MISMATCH);
        return;
    }
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // items (chunk, head) = chunk * H + h over the chunks that exist
    const int total_chunks = p.chunk_off ? p.chunk_off[p.N] : p.N * (int)((p.seq_len + CH - 1) / CH);
    const int n_items = total_chunks * p.H;
    const int q4 = warp & 3, hc = warp >> 2;  // tensor-memory lane quarter, row quarter
    const int L = 32 * q4 + lane;             // this thread's lane: a channel, or a stacked row
    const int c0 = NCOL * hc;                 // first of this thread's 16 rows (or columns)

    unsigned char *sKQ = smem + oKQ, *sV = smem + oV, *sDOY = smem + oDOY, *sS0 = smem + oS0, *sDS = smem + oDS,
                  *sA = smem + oA, *sP = smem + oP, *sU = smem + oU, *sDU = smem + oDU;
    float* fsm = reinterpret_cast<float*>(smem + oSmall);
    float* sInvQ = fsm;
    float* sInvK = sInvQ + nInvQ;
    float* sBeta = sInvK + nInvK;         // [2][64]: beta, then 1 - beta
    float* sFac = sBeta + nBeta;          // [4][64] e^{gc}, e^{gc-ref}, e^{ref-gc}, e^{gT-gc} (Fac order)
    float* sTab = sFac + nFac;            // [6][64] combined row factors (Tab order)
    float* sGate = sTab + nTab;           // gc[64], ref, gT
    // chunk of the current and of the next item, by item parity (seq, local, t0 lo / hi, len)
    int* sCI = reinterpret_cast<int*>(sGate + nGate + 2);
    float* sDgTs = sGate + nGate + nPad;  // [128] state part of dgT
    float* sDgTp = sDgTs + nDgTs;         // [4][128] kr part of dgT per row quarter
    float* sDbP = sDgTp + nDgTp;          // [64] <dY, beta E> per row
    float* sPairR = sDbP + nDbP;          // [4][128] pair-term row sums per column quarter (P rows, then A rows)
    float* sPairC = sPairR + nPairR;      // [4][64] pair-term column sums per lane quarter
    float* sRowG = sPairC + nPairC;       // [4][64] channel sums of the per-element gate terms per lane quarter
    float* sRowQ = sRowG + nRowG;         // [4][64] row dots <dq^, q^> per lane quarter
    float* sRowK = sRowQ + 256;           // [4][64] row dots <dk^, k^>
    float* sTot = sRowQ + nRow;           // [2][64] row dots summed over the lane quarters (q, k)
    uint64_t* mbars = reinterpret_cast<uint64_t*>(sTot + nTot);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbars + 4);
    // operand tiles of an item; MMA completion of the batches with 1, 2 and 3 issuing threads
    const uint32_t mload = smem_u32(mbars), mb1 = smem_u32(mbars + 1), mb2 = smem_u32(mbars + 2),
                   mb3 = smem_u32(mbars + 3);
    const uint32_t mstall = smem_u32(mbars + 5);  // test hook only: a barrier nothing arrives on

    ScalarGates G;
    G.gc = sGate;
    G.ref = sGate + CH;
    G.gT = sGate + CH + 1;

    // the operand tiles of an item: copy `which` (0 .. 9), or all of them (which < 0); k and
    // q are stacked into one 128-row tile, one 64-column box at a time.  The copies may be
    // issued by different threads, at different times and in any order: the barrier's phase
    // cannot complete before the thread of copy 4 (the first one issued) has registered the
    // expectation.
    auto put_ci = [&](int slot, const ChunkInfo& c) {
        int* d = sCI + 8 * slot;
        d[0] = c.seq, d[1] = c.local, d[2] = (int)(c.t0 & 0xffffffff), d[3] = (int)(c.t0 >> 32), d[4] = c.len;
    };
    auto get_ci = [&](int slot) {
        const int* d = sCI + 8 * slot;
        ChunkInfo c;
        c.seq = d[0], c.local = d[1], c.t0 = (int64_t)(((uint64_t)(uint32_t)d[3] << 32) | (uint32_t)d[2]), c.len = d[4];
        return c;
    };
    auto issue_loads = [&](int item, const ChunkInfo& cj, int which) {
        const int hh = item % p.H, hk = qk_head(p, hh), t0 = (int)cj.t0, rcd = item * CH, rdd = item * MD;
        if (which < 0 || which == 4) tc::mbar_expect_tx(mload, 8 * TILE + CH * CH * 2);
        if (which < 0 || which == 0) tc::tma_load_3d(sb + oKQ, &m.k, 0, hk, t0, mload);
        if (which < 0 || which == 1) tc::tma_load_3d(sb + oKQ + 2 * 8192, &m.k, 64, hk, t0, mload);
        if (which < 0 || which == 2) tc::tma_load_3d(sb + oKQ + 8192, &m.q, 0, hk, t0, mload);
        if (which < 0 || which == 3) tc::tma_load_3d(sb + oKQ + 3 * 8192, &m.q, 64, hk, t0, mload);
        if (which < 0 || which == 4) tc::tma_load_4d(sb + oV, &m.v, 0, hh, t0, 0, mload);
        if (which < 0 || which == 5) tc::tma_load_3d(sb + oDOY, &m.dO, 0, hh, t0, mload);
        if (which < 0 || which == 6) tc::tma_load_3d(sb + oDOY + 128 * 128, &m.dO, 64, hh, t0, mload);
        if (which < 0 || which == 7) tc::tma_load_3d(sb + oS0, &m.S0, 0, rdd, 0, mload);
        if (which < 0 || which == 8) tc::tma_load_3d(sb + oDS, &m.dS, 0, rdd, 0, mload);
        if (which < 0 || which == 9) tc::tma_load_2d(sb + oT, &m.T, 0, rcd, mload);
    };

    // ---- set-up: tensor memory, barriers, the first item's loads ----------------------
    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) {
        tc::mbar_init(mload, 1);
        tc::mbar_init(mb1, 1);
        tc::mbar_init(mb2, 2);
        tc::mbar_init(mb3, 3);
        tc::mbar_init(mstall, 1);
        if ((int)blockIdx.x < n_items) {
            ChunkInfo c0i;
            lookup_chunk((int)blockIdx.x / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, c0i);
            put_ci(0, c0i);
            issue_loads(blockIdx.x, c0i, -1);
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    uint32_t phases = 0;  // bit n: the next phase of the barrier with n issuing threads
    int it = 0;                                // this CTA's item count (the load barrier's phase)
    bool pending = (int)blockIdx.x < n_items;  // a load batch is in flight
    uint32_t pend_par = 0;                     // ... on this phase parity of the load barrier
    // the next item's gate (first warp, rows 2 lane and 2 lane + 1) and beta logit (thread
    // r < 64), loaded one item ahead as raw values (rows clamped into the chunk) that are
    // first read at the next item's top, so no thread waits for them
    float pg0 = 0.f, pg1 = 0.f;
    unsigned short pb = 0;
    auto prefetch_small = [&](int item, const ChunkInfo& cj) {
        if (tid >= CH) return;
        const int hh = item % p.H;
        pb = reinterpret_cast<const unsigned short*>(p.beta_logit)[(cj.t0 + min(tid, cj.len - 1)) * p.H + hh];
        if (tid < 32) {
            pg0 = p.g[(cj.t0 + min(2 * tid, cj.len - 1)) * p.H + hh];
            pg1 = p.g[(cj.t0 + min(2 * tid + 1, cj.len - 1)) * p.H + hh];
        }
    };
    if ((int)blockIdx.x < n_items) prefetch_small(blockIdx.x, get_ci(0));
    auto sync_all = [&]() {  // make smem writes visible to the tensor cores and order TMEM use
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    // Waits for the last commit.  If the tensor cores do not answer within the bounded
    // spin, every thread learns it from the vote, the status word records it, the loads
    // in flight are drained (bounded), the tensor memory is released and the CTA returns.
    auto bail = [&]() {
        if (tid == 0) {
            atomicOr(p.status, ST_MMA_TIMEOUT);
            if (pending) tc::mbar_wait(mload, pend_par);
        }
        if (tid == STORE_TID) tc::bulk_wait_all();
        tc::fence_before();
        __syncthreads();
        if (warp == 0) tc::dealloc(tmem, 512);
    };
    auto wait_mma = [&](int n) -> bool {
        const uint32_t bar = n == 1 ? mb1 : n == 2 ? mb2 : mb3;
        const bool ok = tc::mbar_wait(bar, (phases >> n) & 1);
        phases ^= 1u << n;
        tc::fence_after();
        if (__syncthreads_or(!ok)) {
            bail();
            return false;
        }
        return true;
    };
    auto tl = [&](uint32_t col) { return tmem + ((uint32_t)(32 * q4) << 16) + col; };
    auto rows16 = [&](const float* a, float (&o)[16]) {  // a[c0 .. c0+15]
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = *reinterpret_cast<const float4*>(a + c0 + 4 * i);
            o[4 * i] = v.x;
            o[4 * i + 1] = v.y;
            o[4 * i + 2] = v.z;
            o[4 * i + 3] = v.w;
        }
    };
    // row L of a [128][64] bf16 tile, columns c0 .. c0+15, from 16 fp32 values
    auto store_cm = [&](unsigned char* tile, const float (&v)[16]) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, c0 >> 3, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, (c0 >> 3) + 1, 128)) = make_uint4(w[4], w[5], w[6], w[7]);
    };
    // byte offset of element (row c0 + i, column L) in a token-major SW128 tile with `rows` rows
    const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
    auto tok = [&](int rows, int i) -> uint32_t {
        return (uint32_t)((L >> 6) * rows * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
    };
    // raw q (or k) of this thread's channel and rows (staged in tensor memory), and the rows'
    // inverse norms
    auto load_x = [&](bool isq, float (&x)[16], float (&inv)[16]) {
        tc::ld16(tl((isq ? R_Q : R_K) + c0), x);
        rows16(isq ? sInvQ : sInvK, inv);
    };

    // a staged token-major output tile (64 rows x 128 channels, column blocks 8 KB apart) to
    // global memory: one TMA store for a full chunk, else the chunk's valid rows in 16-byte
    // pieces (after a barrier that follows the staging)
    auto put_tile = [&](const CUtensorMap* map, uint32_t tile_off, __nv_bfloat16* dst, const ChunkInfo& c, int hh) {
        if (c.len == CH) {
            if (tid == STORE_TID) {
                tc::tma_store_4d(map, 0, hh, (int)c.t0, 0, sb + tile_off);
                tc::bulk_commit();
            }
        } else {
            for (int i = tid; i < c.len * 16; i += 512) {
                const int r = i >> 4, j = i & 15;
                const uint4 v = *reinterpret_cast<const uint4*>(smem + tile_off + (j >> 3) * 8192 + r * 128 +
                                                                (((j & 7) ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(dst + ((c.t0 + r) * p.H + hh) * MD + j * 8) = v;
            }
        }
    };

    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const int h = item % p.H;
    const ChunkInfo ci = get_ci(it & 1);
    const int next = item + (int)gridDim.x;
    if (tid == 32 && next < n_items) {  // the next item's chunk, for its loads and small values
        ChunkInfo cn;
        lookup_chunk(next / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, cn);
        put_ci((it + 1) & 1, cn);
    }
    if (tid < 32) gdn_gate_scan(2 * tid < ci.len ? pg0 : 0.f, 2 * tid + 1 < ci.len ? pg1 : 0.f, G, false, p);
    if (tid < CH) {  // beta and 1 - beta = sigmoid(-logit) (exact where beta rounds to 1 in fp32)
        const float x = __bfloat162float(__ushort_as_bfloat16(pb));
        sBeta[tid] = tid < ci.len ? sigmoid_f(x) : 0.f;
        sBeta[CH + tid] = tid < ci.len ? sigmoid_f(-x) : 0.f;
    }

    // wait for the operand tiles; rows past the chunk's end are zeroed before any product
    {
        bool ok = tc::mbar_wait(mload, (uint32_t)(it & 1));
        // test hook: the chosen CTA also waits, briefly, on a barrier that no copy, product or
        // thread ever completes, and so takes the same exit as a timed-out wait (its loads in
        // flight have landed: the wait above completed; no product has been issued)
        if (p.test_stall == (int)blockIdx.x + 1 && it == 0 && tid == 0) ok = ok && tc::mbar_wait(mstall, 0, 1 << 12);
        if (__syncthreads_or(!ok)) return bail();
        pending = false;
    }
    if (next < n_items) prefetch_small(next, get_ci((it + 1) & 1));  // first read at the next item's top
    if (ci.len < CH) {
        const int nz = (CH - ci.len) * 16;  // 16-byte chunks per 128-column row
        for (int i = tid; i < 4 * nz; i += 512) {
            const int t = i / nz, rem = i % nz, r = ci.len + rem / 16, jc = rem % 16;
            unsigned char* base = t < 2 ? sKQ : t == 2 ? sV : sDOY;
            const int row = t == 1 ? 64 + r : r, rows = t == 2 ? 64 : 128;
            *reinterpret_cast<uint4*>(base + tc::sw_chunk(row, jc, rows)) = make_uint4(0, 0, 0, 0);
        }
        sync_all();
    }

    // ---- B1: G1 [A; P]_raw = [k; q] k^T, G2 X^T_raw = S0^T k^T, G5b du^T_raw = dS^T k^T:
    //      all on the tiles as loaded, under the prologue below (three issuing threads)
    if (lane == 0 && warp < 3) {
        constexpr uint32_t id1 = tc::idesc(128, 64, 0, 0);
        const uint32_t dst = tmem + (warp == 0 ? R_B : warp == 1 ? R_C : R_G5);
        const uint32_t a = sb + (warp == 0 ? oKQ : warp == 1 ? oS0 : oDS);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(dst, tc::kdesc(a, 128, 0, k), tc::kdesc(sb + oKQ, 128, 0, k), id1, k > 0);
        tc::commit(mb3);
    }

    // ---- prologue, while B1 runs: inverse row norms of q and k (4 threads per row), the
    // gate factor table, the state part of dgT (column sums of the value-major dS . S0),
    // raw q and k of this thread's channel and rows into tensor memory
    {
        const int r = (tid >> 2) & 63, part = tid & 3;
        const int row = tid < 256 ? 64 + r : r;  // q rows, then k rows of the stacked tile
        float s = 0.f;
        for (int jj = 0; jj < 4; ++jj) {
            const int j = tc::rowpart_chunk(part, jj);
            const uint4 v = *reinterpret_cast<const uint4*>(sKQ + tc::sw_chunk(row, j, 128));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16(w[e]);
                s += f.x * f.x + f.y * f.y;
            }
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (part == 0) (tid < 256 ? sInvQ : sInvK)[r] = rsqrtf(s + 1e-6f);
    }
    if (tid < CH) {
        sFac[F_KD * CH + tid] = gate_factor<F_KD>(G, tid);
        sFac[F_KDP * CH + tid] = gate_factor<F_KDP>(G, tid);
        sFac[F_KIP * CH + tid] = gate_factor<F_KIP>(G, tid);
        sFac[F_KR * CH + tid] = gate_factor<F_KR>(G, tid);
    }
    {
        const int cp = tid >> 3, g = tid & 7;  // column pair, row group
        float s0 = 0.f, s1 = 0.f;
        for (int j = g; j < MD; j += 8) {
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
            const float eg = __expf(G.gTv());
            sDgTs[2 * cp] = s0 * eg;
            sDgTs[2 * cp + 1] = s1 * eg;
        }
    }
    {
        float qs[NCOL], ks[NCOL];
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {
            const uint32_t off = tok(128, i);  // k row c0 + i; the q row sits 64 rows (8 KB) below
            ks[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sKQ + off));
            qs[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sKQ + off + 64 * 128));
        }
        tc::st16(tl(R_Q + c0), qs);
        tc::st16(tl(R_K + c0), ks);
    }
    __syncthreads();  // norms and gate factors
    if (tid < CH) {   // combined row factors of the folded products
        const float ik = sInvK[tid], iq = sInvQ[tid], e1 = sFac[F_KDP * CH + tid];
        sTab[T_CF * CH + tid] = ik * sFac[F_KIP * CH + tid];
        sTab[T_KDF * CH + tid] = ik * sFac[F_KD * CH + tid];
        sTab[T_KRF * CH + tid] = ik * sFac[F_KR * CH + tid];
        sTab[T_RA * CH + tid] = sBeta[tid] * ik * e1;
        sTab[T_RP * CH + tid] = p.scale * iq * e1;
        sTab[T_RK * CH + tid] = ik * e1;
    }

    // per-thread accumulators (channel L, rows c0 .. c0+15)
    float dQn[NCOL], dKn[NCOL], dGc[NCOL];
#pragma unroll
    for (int i = 0; i < NCOL; ++i) dQn[i] = dKn[i] = dGc[i] = 0.f;

    // ---- E1: A and P (scaled, masked, bf16), beta E in place of v ----------------------
    if (tid == STORE_TID) tc::bulk_wait_read();  // the last item's dq / dk / dv tiles were read
    if (!wait_mma(3)) return;
    {
        float v[16], cf[16];
        tc::ld16(tl(R_B + c0), v);
        rows16(sTab + T_CF * CH, cf);
        const bool isA = L < 64;  // lanes 0..63: A rows, 64..127: P rows
        const int r = L & 63;
        const float rf = isA ? sTab[T_RA * CH + r] : sTab[T_RP * CH + r];
        unsigned char* dst = isA ? sA : sP;
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i0 = jc * 8 + 2 * e, s0 = c0 + i0;
                float a0 = v[i0] * rf * cf[i0], a1 = v[i0 + 1] * rf * cf[i0 + 1];
                if (isA) {
                    a0 = s0 < r ? a0 : 0.f;
                    a1 = s0 + 1 < r ? a1 : 0.f;
                } else {
                    a0 = s0 <= r ? a0 : 0.f;
                    a1 = s0 + 1 <= r ? a1 : 0.f;
                }
                w[e] = pack_bf16(a0, a1);
            }
            *reinterpret_cast<uint4*>(dst + tc::sw_chunk(r, (c0 >> 3) + jc, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    {
        float v[16], kf[16], bt[16];
        tc::ld16(tl(R_C + c0), v);  // X^T_raw (lane = value channel)
        rows16(sTab + T_KDF * CH, kf);
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // beta E = beta (V - X), in place of V
            __nv_bfloat16* pv = reinterpret_cast<__nv_bfloat16*>(sV + tok(64, i));
            *pv = __float2bfloat16(bt[i] * (__bfloat162float(*pv) - v[i] * kf[i]));
        }
    }
    sync_all();

    // ---- B2: G4 u^T = (beta E)^T T^T ; G5a du^T = dO^T P ------------------------------
    if (lane == 0 && warp < 2) {
        constexpr uint32_t id4 = tc::idesc(128, 64, 1, 0), id5 = tc::idesc(128, 64, 1, 1);
        if (warp == 0) {
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(tmem + R_B, tc::mdesc(sb + oV, 64, 0, k), tc::kdesc(sb + oT, 64, 0, k), id4, k > 0);
        } else {
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(tmem + R_A, tc::mdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oP, 64, 0, k), id5, k > 0);
        }
        tc::commit(mb2);
    }
    if (!wait_mma(2)) return;
    {
        float v[16], w[16], kf[16];
        tc::ld16(tl(R_B + c0), v);
        store_cm(sU, v);  // u^T [j][r]
        tc::ld16(tl(R_A + c0), v);
        tc::ld16(tl(R_G5 + c0), w);
        rows16(sTab + T_KRF * CH, kf);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) {  // + dS^T kr^T
            const float2 r = __ffma2_rn(F2(w, i), F2(kf, i), F2(v, i));
            v[i] = r.x, v[i + 1] = r.y;
        }
        store_cm(sDU, v);  // du^T [j][r]
    }
    sync_all();

    // ---- B3: G6 dY^T = du^T T ; dv = beta dY, dY into the lower half of [dO; dY] ---------
    if (tid == 0) {
        constexpr uint32_t id6 = tc::idesc(128, 64, 0, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oDU, 128, 0, k), tc::mdesc(sb + oT, 64, 0, k), id6, k > 0);
        tc::commit(mb1);
    }
    if (!wait_mma(1)) return;
    {
        float v[16], bt[16];
        tc::ld16(tl(R_D + c0), v);
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {
            *reinterpret_cast<__nv_bfloat16*>(sDU + tok(64, i)) = __float2bfloat16(bt[i] * v[i]);  // dv, staged
            *reinterpret_cast<__nv_bfloat16*>(sDOY + tok(128, i) + 64 * 128) = __float2bfloat16(v[i]);  // dY
        }
    }
    sync_all();
    put_tile(&m.dv, oDU, p.dv, ci, h);

    // ---- B4: G3/G7 [dqd^T, Z^T] = S0 [dO; dY]^T ; G8 dkr^T = dS u^T ; G9 [dP; dA]_raw =
    //      [dO; dY] u^T (three issuing threads)
    if (lane == 0 && warp < 3) {
        if (warp == 0) {
            constexpr uint32_t id37 = tc::idesc(128, 128, 1, 0);
#pragma unroll
            for (int k = 0; k < MD; k += 16)
                tc::mma(tmem + R_A, tc::mdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oDOY, 128, 0, k), id37, k > 0);
        } else if (warp == 1) {
            constexpr uint32_t id8 = tc::idesc(128, 64, 1, 1);
#pragma unroll
            for (int k = 0; k < MD; k += 16)
                tc::mma(tmem + R_C, tc::mdesc(sb + oDS, 128, 0, k), tc::mdesc(sb + oU, 128, 0, k), id8, k > 0);
        } else {
            constexpr uint32_t id9 = tc::idesc(128, 64, 0, 1);
#pragma unroll
            for (int k = 0; k < MD; k += 16)
                tc::mma(tmem + R_D, tc::kdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oU, 128, 0, k), id9, k > 0);
        }
        tc::commit(mb3);
    }
    // while the tensor cores run: <dY, beta E> per row (token-major, 4 threads per row)
    if (tid < 4 * CH) {
        const int r = tid >> 2, part = tid & 3;
        float s2 = 0.f;
        for (int jj = 0; jj < 4; ++jj) {
            const int j = tc::rowpart_chunk(part, jj);
            const uint4 a = *reinterpret_cast<const uint4*>(sDOY + tc::sw_chunk(64 + r, j, 128));
            const uint4 b = *reinterpret_cast<const uint4*>(sV + tc::sw_chunk(r, j, 64));
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
    if (!wait_mma(3)) return;
    // v, dO, S0 and T are dead: the next item's copies of them start now (k, q, dS after B5)
    if (next < n_items) {
        if (lane == 0 && warp < 5) issue_loads(next, get_ci((it + 1) & 1), warp == 0 ? 4 : warp == 4 ? 9 : warp + 4);
        pending = true;
        pend_par = (uint32_t)((it + 1) & 1);
    }
    {
        float v[16], f[16], x[16], inv[16], bt[16];
        rows16(sFac + F_KD * CH, f);
        tc::ld16(tl(R_A + c0), v);  // dqd^T (lane = key channel)
        load_x(true, x, inv);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) {  // dqd
            const float2 t = __fmul2_rn(__fmul2_rn(make_float2(p.scale, p.scale), F2(v, i)), F2(f, i));
            ACC2(dQn, i, __fadd2_rn(F2(dQn, i), t));
            ACC2(dGc, i, __ffma2_rn(__fmul2_rn(F2(x, i), F2(inv, i)), t, F2(dGc, i)));
        }
        tc::ld16(tl(R_A + 64 + c0), v);  // Z^T
        load_x(false, x, inv);
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) {  // dkd (from E) = -beta Z
            const float2 t = __fmul2_rn(__fmul2_rn(make_float2(-bt[i], -bt[i + 1]), F2(v, i)), F2(f, i));
            ACC2(dKn, i, __fadd2_rn(F2(dKn, i), t));
            ACC2(dGc, i, __ffma2_rn(__fmul2_rn(F2(x, i), F2(inv, i)), t, F2(dGc, i)));
        }
        tc::ld16(tl(R_C + c0), v);
        rows16(sFac + F_KR * CH, f);
        float2 dgt2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) {  // dkr
            const float2 t = __fmul2_rn(F2(v, i), F2(f, i));
            ACC2(dKn, i, __fadd2_rn(F2(dKn, i), t));
            const float2 kt = __fmul2_rn(__fmul2_rn(F2(x, i), F2(inv, i)), t);
            ACC2(dGc, i, __fadd2_rn(F2(dGc, i), make_float2(-kt.x, -kt.y)));
            dgt2 = __fadd2_rn(dgt2, kt);
        }
        const float dgt = dgt2.x + dgt2.y;
        sDgTp[hc * MD + L] = dgt;
    }
    {
        // lanes 0..63: dP rows, lanes 64..127: dA rows.  Pair terms t = dP P (s <= r) and
        // dA A (s < r); X10 = [dP; beta dA] x invk_s e^{ref-gc_s} (column s), X11 = [dP x scale
        // invq_r e^{gc_r-ref}; beta dA x invk_r e^{gc_r-ref}] (row r), into the dS space
        float v[16], t[16];
        tc::ld16(tl(R_D + c0), v);
        const bool isP = L < 64;
        const int r = L & 63;
        const unsigned char* src = isP ? sP : sA;
        float rs = 0.f;
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            const uint4 av = *reinterpret_cast<const uint4*>(src + tc::sw_chunk(r, (c0 >> 3) + jc, 64));
            const uint32_t wa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i0 = jc * 8 + 2 * e, s0 = c0 + i0;
                float a0 = v[i0], a1 = v[i0 + 1];
                if (isP) {
                    a0 = s0 <= r ? a0 : 0.f;
                    a1 = s0 + 1 <= r ? a1 : 0.f;
                } else {
                    a0 = s0 < r ? -a0 : 0.f;
                    a1 = s0 + 1 < r ? -a1 : 0.f;
                }
                const float2 pe = unpack_bf16(wa[e]);
                t[i0] = a0 * pe.x;
                t[i0 + 1] = a1 * pe.y;
                rs += t[i0];
                rs += t[i0 + 1];
                v[i0] = a0;
                v[i0 + 1] = a1;
            }
        }
        sPairR[hc * 128 + L] = rs;
        const float cs = warp_transpose_sum16(t);  // lanes 2i, 2i + 1: column c0 + i over this warp's rows
        if ((lane & 1) == 0) sPairC[q4 * CH + c0 + (lane >> 1)] = cs;
        const float br = isP ? 1.f : sBeta[r];
        float o[16], cf[16];
        rows16(sTab + T_CF * CH, cf);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) ACC2(o, i, __fmul2_rn(__fmul2_rn(make_float2(br, br), F2(v, i)), F2(cf, i)));
        store_cm(sDS, o);
        const float rf = isP ? sTab[T_RP * CH + r] : br * sTab[T_RK * CH + r];
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) ACC2(o, i, __fmul2_rn(F2(v, i), make_float2(rf, rf)));
        store_cm(sDS + TILE, o);
    }
    sync_all();

    // ---- B5: G10 [dqd', dkd']^T = k^T X10^T ; G11 dki'^T = q^T X11_P + k^T X11_A ----------
    if (lane == 0 && warp < 2) {
        if (warp == 0) {
            constexpr uint32_t id10 = tc::idesc(128, 128, 1, 0);
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(tmem + R_A, tc::mdesc(sb + oKQ, 128, 0, k), tc::kdesc(sb + oDS, 128, 0, k), id10, k > 0);
        } else {
            constexpr uint32_t id11 = tc::idesc(128, 64, 1, 1);
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(tmem + R_B, tc::mdesc(sb + oKQ, 128, 64, k), tc::mdesc(sb + oDS + TILE, 128, 0, k), id11, k > 0);
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(tmem + R_B, tc::mdesc(sb + oKQ, 128, 0, k), tc::mdesc(sb + oDS + TILE, 128, 64, k), id11, 1);
        }
        tc::commit(mb2);
    }
    if (!wait_mma(2)) return;
    // every large shared tile is dead: the rest of the next item's operands
    if (next < n_items && lane == 0 && warp < 5)
        issue_loads(next, get_ci((it + 1) & 1), warp == 4 ? 8 : warp);
    {
        float f[16], v[16];
        rows16(sFac + F_KDP * CH, f);
        tc::ld16(tl(R_A + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2)  // dqd'
            ACC2(dQn, i, __ffma2_rn(__fmul2_rn(make_float2(p.scale, p.scale), F2(v, i)), F2(f, i), F2(dQn, i)));
        tc::ld16(tl(R_A + 64 + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) ACC2(dKn, i, __ffma2_rn(F2(v, i), F2(f, i), F2(dKn, i)));  // dkd'
        rows16(sFac + F_KIP * CH, f);
        tc::ld16(tl(R_B + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; i += 2) ACC2(dKn, i, __ffma2_rn(F2(v, i), F2(f, i), F2(dKn, i)));  // dki'
    }

    // ---- epilogue: L2-norm backward, dq / dk, dbeta, the gate gradient ----------------------
    {  // channel sums of the per-element gate terms per row (dGc is dead afterwards)
        const float sg = warp_transpose_sum16(dGc);  // lanes 2i, 2i+1: row c0 + i
        if ((lane & 1) == 0) sRowG[q4 * CH + c0 + (lane >> 1)] = sg;
    }
    {
        // per-row dots over this warp's 32 channels: lane l gets row c0 + (l & 15)
        float t[32];
        {
            float x[16], inv[16];
            load_x(true, x, inv);
#pragma unroll
            for (int i = 0; i < NCOL; i += 2) ACC2(t, i, __fmul2_rn(__fmul2_rn(F2(dQn, i), F2(x, i)), F2(inv, i)));
            load_x(false, x, inv);
#pragma unroll
            for (int i = 0; i < NCOL; i += 2) ACC2(t, 16 + i, __fmul2_rn(__fmul2_rn(F2(dKn, i), F2(x, i)), F2(inv, i)));
        }
        const float s = warp_transpose_sum32(t);  // lane l: value l (l < 16: q row c0+l, else k row c0+l-16)
        (lane < 16 ? sRowQ : sRowK)[q4 * CH + c0 + (lane & 15)] = s;
    }
    __syncthreads();
    if (tid < 2 * CH) {  // sums over the four lane quarters, once per row
        const float* part = tid < CH ? sRowQ : sRowK;
        const int r = tid & (CH - 1);
        sTot[tid] = ((part[r] + part[CH + r]) + part[2 * CH + r]) + part[3 * CH + r];
    }
    __syncthreads();
    {
        // dq into the dead u^T tile, dk into the dead A and P tiles (one 16 KB token-major
        // tile), or row by row for a chunk cut by its sequence's end
        float x[16], inv[16], tt[16];
        load_x(true, x, inv);
        rows16(sTot, tt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i)
            *reinterpret_cast<__nv_bfloat16*>(sU + tok(64, i)) =
                __float2bfloat16((dQn[i] - x[i] * inv[i] * tt[i]) * inv[i]);
        load_x(false, x, inv);
        rows16(sTot + CH, tt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i)
            *reinterpret_cast<__nv_bfloat16*>(sA + tok(64, i)) =
                __float2bfloat16((dKn[i] - x[i] * inv[i] * tt[i]) * inv[i]);
    }
    tc::fence_async_smem();  // the staged dq / dk reach the copy engine after the next barrier
    // dbeta (logit space): <dY, beta E> + rowsum(dA . A)
    for (int r = tid; r < ci.len; r += 512) {
        const float dA_A = ((sPairR[CH + r] + sPairR[128 + CH + r]) + sPairR[256 + CH + r]) + sPairR[384 + CH + r];
        p.dbeta[(ci.t0 + r) * p.H + h] = __float2bfloat16(sBeta[CH + r] * (sDbP[r] + dA_A));
    }
    // dg: per row, the channel sums of the per-element terms plus the pair terms (row sums
    // minus column sums), suffix sums over the rows, plus the chunk constant dgT
    if (warp == 0) {
        auto dgT_of = [&](int d) -> float {
            return (((sDgTs[d] + sDgTp[d]) + sDgTp[MD + d]) + sDgTp[2 * MD + d]) + sDgTp[3 * MD + d];
        };
        auto row_total = [&](int r) -> float {
            const float el = ((sRowG[r] + sRowG[CH + r]) + sRowG[2 * CH + r]) + sRowG[3 * CH + r];
            const float pr = ((sPairR[r] + sPairR[128 + r]) + sPairR[256 + r]) + sPairR[384 + r];
            const float ar = ((sPairR[CH + r] + sPairR[128 + CH + r]) + sPairR[256 + CH + r]) + sPairR[384 + CH + r];
            const float pc = ((sPairC[r] + sPairC[CH + r]) + sPairC[2 * CH + r]) + sPairC[3 * CH + r];
            return el + ((pr + ar) - pc);
        };
        float t = 0.f;
        for (int d = lane; d < MD; d += 32) t += dgT_of(d);
        t = warp_sum(t);
        const int r0 = 2 * lane;
        const float a = row_total(r0), b = row_total(r0 + 1);
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
    __syncthreads();  // this item's small arrays and tensor memory are free
    tc::fence_after();
    put_tile(&m.dq, oU, p.dq, ci, h);
    put_tile(&m.dk, oA, p.dk, ci, h);
    }
    if (tid == STORE_TID) tc::bulk_wait_all();
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_main_gdn(const Params& p, cudaStream_t s) {
    GdnMaps m;
    const uint64_t rows_cc = (uint64_t)p.max_chunks * p.H * CH;
    const uint64_t rows_dd = (uint64_t)p.max_chunks * p.H * MD;
    const uint64_t T = (uint64_t)p.T_total;
    bool ok = encode_tokens_map(&m.q, p.q, T, p.Hk, MD) && encode_tokens_map(&m.k, p.k, T, p.Hk, MD) &&
              encode_blocked_tokens_map(&m.v, p.v, T, p.H) && encode_tokens_map(&m.dO, p.dO, T, p.H, MD) &&
              encode_blocked_rows_map(&m.S0, p.S0, rows_dd, MD) && encode_blocked_rows_map(&m.dS, p.dS, rows_dd, MD) &&
              encode_rows_map(&m.T, p.Tm, rows_cc, CH, CH) && encode_blocked_tokens_map(&m.dq, p.dq, T, p.H) &&
              encode_blocked_tokens_map(&m.dk, p.dk, T, p.H) && encode_blocked_tokens_map(&m.dv, p.dv, T, p.H);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_main_gdn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int items = p.max_chunks * p.H;
    const int ctas = items < num_sms() ? items : num_sms();
    k_main_gdn<<<ctas, 512, SMEM_BYTES, s>>>(p, m);
    return cudaGetLastError();
}

}  // namespace gdr
