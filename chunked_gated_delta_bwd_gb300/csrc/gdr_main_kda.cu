// Chunk-parallel main backward on tcgen05 for D = 128 with the per-channel (KDA) gate:
// persistent CTAs of 16 warps, one per SM, each looping over (chunk, head) items; the
// next item's operand tiles arrive by TMA while the current item's epilogue runs (every
// large shared tile is dead after the last product group).  The scalar gate has its
// own kernel, gdr_main_gdn.cu.  Every product is a 128-row tcgen05 MMA into tensor memory, written feature-major
// where the natural output is C x D: the accumulator holds X^T (lane = key channel d
// or value channel j, column = token row r), so a thread owns one channel for 16
// rows.  The raw q and k rows and e^{gc - ref} of the per-channel cumulative gate gc
// are staged in tensor memory in that layout once, and every derived tile (kd', ki',
// qd', kd, kr) is built from registers, channel-major ([d][r]), with 16-byte stores.
//
// With S0 = chunk-start state, dS = state gradient at the chunk end (both value-major
// [j][d]) and [X; Y] a 128-row operand stacked from two 64-row tiles:
//   G1  [A_raw; P]   = [kd'; qd'] ki'^T  (computed by the prep kernel, which needs A for the
//                      inverse: A = beta A_raw and P (a bf16 pair) arrive by TMA)
//                                                       G7  Z^T    = S0 dY^T
//   G2  X^T          = S0^T kd^T                        G8  dkr^T  = dS u^T
//   G3  dqd^T        = S0 dO^T                          G9  [dP; dA] = [dO; dY] u^T
//   G4  u^T          = (beta E)^T T^T                   G10 [dqd', dkd']^T = ki'^T [dP; beta dA]^T
//   G5  du^T         = dO^T P + dS^T kr^T               G11 dki'^T = qd'^T dP + kd'^T (beta dA)
//   G6  dY^T         = du^T T
// followed by the elementwise assembly of "FlashKDA之backward（K1）" (§3.2-§3.3, §5).
//
// dv, dq, dk and dg_raw are staged token-major in shared tiles that are dead by then
// (du^T, ki' lo, the dY rows of [dO; dY], the raw-gate tile) and written by TMA stores; a
// chunk cut by its sequence's end copies its valid rows from the staged tile instead.
//
// KDA runs in precise mode: the operands that carry the
// per-channel gate gradient (beta E, u, dP and beta dA, and ki', qd', kd' of G10 / G11)
// are bf16 pairs hi + lo and each of those products is hi*hi + lo*hi + hi*lo, and P is a
// pair in G5a (dO^T P_hi + dO^T P_lo), because dA_log and ddt_bias sum dg over every token
// of a head.
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"

namespace gdr {

namespace {

constexpr int MD = 128;
constexpr int TILE = CH * MD * 2;  // 16 KB: a C x D token-major or a D x C channel-major bf16 tile
// shared-memory map (bytes from the 1024-aligned base); later tenants after the arrows
constexpr int oK = 0;           // k (token-major)     -> kr [d][r] -> beta E lo -> qd' lo
constexpr int oV = 16384;       // v -> beta E (token-major)
constexpr int oDOY = 32768;     // [dO; dY] token-major, 128 rows
constexpr int oS0 = 65536;      // S0 [j][d]          -> kd' [d][r] (+ lo at +16 KB)
constexpr int oDS = 98304;      // dS [j][d]          -> [dP; beta dA] [m][s] (+ lo at +16 KB)
constexpr int oT = 131072;      // T  [r][s]
constexpr int oA = 139264;      // A = beta A_raw, strict lower [r][s] (prep) -> raw gate tile, with P's space
constexpr int oP = 147456;      // P, lower [r][s] (prep)
constexpr int oW0 = 155648;     // raw gate tile -> kd [d][r] -> u^T lo -> ki' [d][r]
constexpr int oW1 = 172032;     // u^T [j][r] -> ki' lo -> dq (staged)
constexpr int oW2 = 188416;     // q (token-major) -> du^T -> dv (staged) -> qd' [d][r]
constexpr int oPL = 204800;     // P lo: the residual P - bf16(P), the pair's second half (prep; G5a)
constexpr int oSmall = oPL + 8192;
// small arrays (floats)
constexpr int NCOL = 16;  // rows per thread (16 warps: 4 lane quarters x 4 row quarters)
constexpr int nInvQ = 64, nInvK = 64, nBeta = 128, nFac = 256, nGate = 128, nRef = 128, nGT = 128,
              nScan = 512, nDgTs = 128, nDgTp = 512, nDbP = 64, nDbA = 256, nRow = 512, nMisc = 64, nTot = 128;
constexpr int SMALL_FLOATS =
    nInvQ + nInvK + nBeta + nFac + nGate + nRef + nGT + nScan + nDgTs + nDgTp + nDbP + nDbA + nRow + nMisc + nTot;
constexpr int SMEM_BYTES = oSmall + SMALL_FLOATS * 4 + 64 + 1024;  // + mbarriers / tmem slot + alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// tensor-memory columns
constexpr uint32_t R_A = 0, R_B = 128, R_C = 192, R_D = 256, R_Q = 320, R_K = 384, R_G = 448;

struct MainMaps {
    CUtensorMap q, k, v, dO, S0, dS, T, ap, graw, dq, dk, dv, dgr;
};
constexpr int STORE_TID = 96;  // the thread that issues the TMA stores of dq, dk, dv and dg_raw

}  // namespace

template <int GATE>
__global__ void __launch_bounds__(512, 1) k_main_kda(const Params p, const __grid_constant__ MainMaps m) {
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
    const int c0 = NCOL * hc;                 // first of this thread's 16 rows

    unsigned char *sK = smem + oK, *sV = smem + oV, *sDOY = smem + oDOY, *sS0 = smem + oS0, *sDS = smem + oDS,
                  *sA = smem + oA, *sW0 = smem + oW0, *sW1 = smem + oW1, *sW2 = smem + oW2;
    float* fsm = reinterpret_cast<float*>(smem + oSmall);
    float* sInvQ = fsm;
    float* sInvK = sInvQ + nInvQ;
    float* sBeta = sInvK + nInvK;         // [2][64]: beta, then 1 - beta
    float* sFac = sBeta + nBeta;     // [2][128]: e^{ref}, e^{gT-ref} per channel
    float* sGate = sFac + nFac;      // dt_bias[d]
    float* sRef = sGate + nGate;     // ref[d]
    float* sGT = sRef + nRef;        // gT[d]
    float* sScan = sGT + nGT;        // [4][128] per-quarter gate totals / extrema / suffix totals
    float* sDgTs = sScan + nScan;    // [128] state part of dgT
    float* sDgTp = sDgTs + nDgTs;    // [4][128] kr part of dgT per row quarter
    float* sDbP = sDgTp + nDgTp;     // [64] <dY, beta E> per row
    float* sDbA = sDbP + nDbP;       // [4][64] rowsum(dA . A) per column quarter
    float* sRow = sDbA + nDbA;       // [2][4][64] row dots; earlier the [4][128] per-quarter gate minima
    float* sMisc = sRow + nRow;      // [64]: per-warp partials [0, 16); e^{A_log} at [32]; chunk slots at [48, 64)
    float* sTot = sMisc + nMisc;     // [2][64] row dots summed over the lane quarters (q, k)
    uint64_t* mbars = reinterpret_cast<uint64_t*>(sTot + nTot);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbars + 4);
    // MMA completion; operand tiles of an item; the raw gate tile for the gate chain rule; the
    // item's A and P pair from the prep kernel
    const uint32_t mb = smem_u32(mbars), mload = smem_u32(mbars + 1), mgr = smem_u32(mbars + 2),
                   mAP = smem_u32(mbars + 3);

    // chunk of the current and of the next item, by item parity (seq, local, t0 lo / hi, len):
    // the next item's is looked up by one thread at the top of an item, so no thread waits for
    // the chunk table where the next item's copies are requested
    int* sCI = reinterpret_cast<int*>(sMisc + 48);
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
    // the operand tiles of an item: copy `which` (0 .. 8), or all of them (which < 0).  The
    // copies may be issued by different threads and in any order: the transaction count of
    // the barrier can run ahead of the expectation that copy 0's thread registers.
    auto issue_loads = [&](int item, const ChunkInfo& cj, int which) {
        const int hh = item % p.H, t0 = (int)cj.t0, rcd = item * CH, rdd = item * MD;
        if (which <= 0) tc::mbar_expect_tx(mload, 4 * TILE + 2 * 2 * TILE + CH * CH * 2 + TILE);
        if (which < 0 || which == 0)
            tc::tma_load_4d(sb + oW0, &m.graw, 0, hh, t0, 0, mload);  // raw gates (token-major)
        if (which < 0 || which == 1) tc::tma_load_4d(sb + oK, &m.k, 0, qk_head(p, hh), t0, 0, mload);
        if (which < 0 || which == 2) tc::tma_load_4d(sb + oV, &m.v, 0, hh, t0, 0, mload);
        if (which < 0 || which == 3) tc::tma_load_4d(sb + oW2, &m.q, 0, qk_head(p, hh), t0, 0, mload);
        if (which < 0 || which == 4)  // rows 0..63 of a 128-row tile
            tc::tma_load_3d(sb + oDOY, &m.dO, 0, hh, t0, mload);
        if (which < 0 || which == 5) tc::tma_load_3d(sb + oDOY + 128 * 128, &m.dO, 64, hh, t0, mload);
        if (which < 0 || which == 6) tc::tma_load_3d(sb + oS0, &m.S0, 0, rdd, 0, mload);
        if (which < 0 || which == 7) tc::tma_load_3d(sb + oDS, &m.dS, 0, rdd, 0, mload);
        if (which < 0 || which == 8) tc::tma_load_2d(sb + oT, &m.T, 0, rcd, mload);
    };

    // ---- set-up: tensor memory, barriers, the first item's loads ----------------------
    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) {
        tc::mbar_init(mb, 1);
        tc::mbar_init(mload, 1);
        tc::mbar_init(mgr, 1);
        tc::mbar_init(mAP, 1);
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
    uint32_t phase = 0;
    int it = 0;              // this CTA's item count (the load barrier's phase)
    bool pending = (int)blockIdx.x < n_items;  // a load batch is in flight
    uint32_t pend_par = 0;                     // ... on this phase parity of the load barrier
    bool pending_g = false;                    // a raw gate tile is in flight
    bool pending_ap = false;                   // the item's A and P pair are in flight
    // the next item's beta logit (thread r < 64, a raw value, row clamped into the chunk) and
    // gate parameters, loaded one item ahead and first read at the next item's top, so no
    // thread waits for them
    unsigned short pb = 0;
    float palog = 0.f, pbias = 0.f;  // the next item's gate parameters (this thread's channel)
    auto prefetch_small = [&](int item, const ChunkInfo& cj) {
        const int hh = item % p.H;
        palog = p.A_log[hh];
        pbias = p.dt_bias[hh * MD + L];
        if (tid >= CH) return;
        pb = reinterpret_cast<const unsigned short*>(p.beta_logit)[(cj.t0 + min(tid, cj.len - 1)) * p.H + hh];
    };
    if ((int)blockIdx.x < n_items) prefetch_small(blockIdx.x, get_ci(0));
    auto sync_all = [&]() {  // make smem writes visible to the tensor cores and order TMEM use
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    // Waits for the last commit.  If the tensor cores do not answer within the
    // bounded spin, every thread learns it from the vote, the status word records
    // it, the tensor memory is released and the CTA returns.
    auto bail = [&]() {
        if (tid == 0) {
            atomicOr(p.status, ST_MMA_TIMEOUT);
            if (pending) tc::mbar_wait(mload, pend_par);  // bounded drain of the loads in flight
            if (pending_g) tc::mbar_wait(mgr, (uint32_t)(it & 1));
            if (pending_ap) tc::mbar_wait(mAP, (uint32_t)(it & 1));
        }
        if (tid == STORE_TID) tc::bulk_wait_all();
        tc::fence_before();
        __syncthreads();
        if (warp == 0) tc::dealloc(tmem, 512);
    };
    auto wait_mma = [&]() -> bool {
        const bool ok = tc::mbar_wait(mb, phase);
        phase ^= 1;
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
    // row L of a channel-major [128][64] tile, columns c0 .. c0+15, from 16 fp32 values
    auto store_cm = [&](unsigned char* tile, const float (&v)[16]) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, c0 >> 3, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, (c0 >> 3) + 1, 128)) = make_uint4(w[4], w[5], w[6], w[7]);
    };
    // the same as a bf16 pair: hi to `tile`, the residual v - hi to `lo`
    auto store_cm_pair = [&](unsigned char* tile, unsigned char* lo, const float (&v)[16]) {
        uint32_t w[8], wl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            w[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
            const float2 hf = unpack_bf16(w[e]);
            wl[e] = pack_bf16(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
        }
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, c0 >> 3, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, (c0 >> 3) + 1, 128)) = make_uint4(w[4], w[5], w[6], w[7]);
        *reinterpret_cast<uint4*>(lo + tc::sw_chunk(L, c0 >> 3, 128)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        *reinterpret_cast<uint4*>(lo + tc::sw_chunk(L, (c0 >> 3) + 1, 128)) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
    };

    // a staged token-major output tile (64 rows x 128 channels; the column blocks `bstride`
    // bytes apart) to global memory: one TMA store (4D map: blocks 8 KB apart; 3D map: one
    // store per block) for a full chunk, else the chunk's valid rows in 16-byte pieces
    auto put_tile = [&](const CUtensorMap* map, bool blocked, uint32_t tile_off, int bstride, __nv_bfloat16* dst,
                        const ChunkInfo& c, int hh) {
        if (c.len == CH) {
            if (tid == STORE_TID) {
                if (blocked) {
                    tc::tma_store_4d(map, 0, hh, (int)c.t0, 0, sb + tile_off);
                } else {
                    tc::tma_store_3d(map, 0, hh, (int)c.t0, sb + tile_off);
                    tc::tma_store_3d(map, 64, hh, (int)c.t0, sb + tile_off + bstride);
                }
                tc::bulk_commit();
            }
        } else {
            for (int i = tid; i < c.len * 16; i += 512) {
                const int r = i >> 4, j = i & 15;
                const uint4 v = *reinterpret_cast<const uint4*>(smem + tile_off + (j >> 3) * bstride + r * 128 +
                                                                (((j & 7) ^ (r & 7)) << 4));
                *reinterpret_cast<uint4*>(dst + ((c.t0 + r) * p.H + hh) * MD + j * 8) = v;
            }
        }
    };

    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const int h = item % p.H;
    const ChunkInfo ci = get_ci(it & 1);
    if (tid == 32 && item + (int)gridDim.x < n_items) {  // the next item's chunk
        ChunkInfo cn;
        lookup_chunk((item + (int)gridDim.x) / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, cn);
        put_ci((it + 1) & 1, cn);
    }
    if (tid < CH) {  // beta and 1 - beta = sigmoid(-logit) (exact where beta rounds to 1 in fp32)
        const float x = __bfloat162float(__ushort_as_bfloat16(pb));
        sBeta[tid] = tid < ci.len ? sigmoid_f(x) : 0.f;
        sBeta[CH + tid] = tid < ci.len ? sigmoid_f(-x) : 0.f;
    }
    const float alog = palog, bias = pbias;  // gate parameters, loaded one item ahead

    // wait for the operand tiles; rows past the chunk's end read as zero
    {
        const bool ok = tc::mbar_wait(mload, (uint32_t)(it & 1));
        if (__syncthreads_or(!ok)) return bail();
        pending = false;
    }
    // per-channel log gates of this thread's channel and rows, scanned across the four
    // row quarters; once the chunk's reference is known, e^{gc - ref} is staged in tensor
    // memory (lane = channel, column = row) and the other gate factors derive from it
    float g[16];  // cumulative gates of this thread's rows
    const float a = expf(alog);
    if (hc == 0) sGate[L] = bias;  // for the gate chain rule at the end of the item
    if (tid == 0) sMisc[32] = a;
    {
        const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
            g[i] = c0 + i < ci.len ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sW0 + off)) : 0.f;
        }
    }
    // the quarter's scan, its total and extrema; one exchange gives every thread the
    // prefix, the chunk total and the chunk's extrema of its channel (the maximum over the
    // rows is the largest quarter maximum plus that quarter's prefix: fp32 addition is
    // monotone, so this is the maximum of the prefixed values bit for bit)
    float acc = 0.f, lmx = -3.0e38f, lmn = 3.0e38f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (c0 + i < ci.len) acc += kda_gate_fn<GATE>(p.gate_scale, a, g[i] + bias);
        g[i] = acc;
        lmx = fmaxf(lmx, acc);
        lmn = fminf(lmn, acc);
    }
    // (sRow holds the row dots later in the item and sDgTp the kr part of dgT: both free here)
    sScan[hc * MD + L] = acc;
    sRow[hc * MD + L] = lmx;
    sDgTp[hc * MD + L] = lmn;
    __syncthreads();
    if (tid == STORE_TID) {
        // the item's A and the P pair (written by the prep kernel) into the A, P and P-lo
        // tiles: dead since the last item's dg_raw store read them (A, P) and its G5a (P lo);
        // first needed by G5a, several thousand cycles from here
        tc::bulk_wait_read();
        tc::mbar_expect_tx(mAP, 3 * CH * CH * 2);
        tc::tma_load_2d(sb + oA, &m.ap, 0, 3 * item * CH, mAP);
        tc::tma_load_2d(sb + oP, &m.ap, 0, (3 * item + 1) * CH, mAP);
        tc::tma_load_2d(sb + oPL, &m.ap, 0, (3 * item + 2) * CH, mAP);
    }
    pending_ap = true;
    float pre = 0.f, tot = 0.f, M = -3.0e38f, N = 3.0e38f;
#pragma unroll
    for (int h2 = 0; h2 < 4; ++h2) {
        const float t = sScan[h2 * MD + L];
        M = fmaxf(M, tot + sRow[h2 * MD + L]);
        N = fminf(N, tot + sDgTp[h2 * MD + L]);
        if (h2 < hc) pre += t;
        tot += t;
    }
    const float refL = 0.5f * (M + N);
    float f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __expf((g[i] + pre) - refL);
    tc::st16(tl(R_G + c0), f);
    if (hc == 0) {
        sRef[L] = refL;
        sGT[L] = tot;
        sFac[L] = __expf(refL);             // e^{ref}
        sFac[MD + L] = __expf(tot - refL);  // e^{gT - ref}
    }

    if (ci.len < CH) {
        const int nz = (CH - ci.len) * 16;  // 16-byte chunks per 64-row tile (2 blocks x 8)
        for (int i = tid; i < 4 * nz; i += 512) {
            const int t = i / nz, rem = i % nz, r = ci.len + rem / 16, jc = rem % 16;
            unsigned char* base = t == 0 ? sK : t == 1 ? sV : t == 2 ? sW2 : sDOY;
            const int rows = t == 3 ? 128 : 64;
            *reinterpret_cast<uint4*>(base + tc::sw_chunk(r, jc, rows)) = make_uint4(0, 0, 0, 0);
        }
    }
    __syncthreads();

    // inverse row norms of q (from W2) and k, 4 threads per row;
    // dgT state part (column sums of the value-major dS . S0)
    {
        const int r = (tid >> 2) & 63, part = tid & 3;
        const unsigned char* src = tid < 256 ? sW2 : sK;
        float s = 0.f;
        for (int jj = 0; jj < 4; ++jj) {
            const int j = tc::rowpart_chunk(part, jj);
            const uint4 v = *reinterpret_cast<const uint4*>(src + tc::sw_chunk(r, j, 64));
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
            sDgTs[2 * cp] = s0 * __expf(sGT[2 * cp]);
            sDgTs[2 * cp + 1] = s1 * __expf(sGT[2 * cp + 1]);
        
        }
    }
    // raw q and k of this thread's channel and rows into tensor memory
    {
        const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
        float qs[NCOL], ks[NCOL];
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {
            const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
            qs[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sW2 + off));
            ks[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sK + off));
        }
        tc::st16(tl(R_Q + c0), qs);
        tc::st16(tl(R_K + c0), ks);
    }
    if (tid == STORE_TID) tc::bulk_wait_read();  // the last item's staged outputs were read
    __syncthreads();  // norms, factors and the q tile reads are done

    // per-element factors of this thread's channel and rows
    auto factors = [&](int kind, float (&f)[16]) {
        // e^{gc-ref} from tensor memory; e^{gc} = e^{gc-ref} e^{ref}, e^{ref-gc} = 1 / e^{gc-ref},
        // e^{gT-gc} = e^{gT-ref} / e^{gc-ref} (|gc - ref| <= 80: no overflow)
        const float eRef = sFac[L], eGTref = sFac[MD + L];
        float e[16];
        tc::ld16(tl(R_G + c0), e);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (kind == F_KDP) f[i] = e[i];
            else if (kind == F_KD) f[i] = e[i] * eRef;
            else if (kind == F_KIP) f[i] = __fdividef(1.f, e[i]);
            else f[i] = __fdividef(eGTref, e[i]);
        }
    
    };
    // raw q (or k) of this thread's channel and rows, and the rows' inverse norms
    auto load_x = [&](bool isq, float (&x)[16], float (&inv)[16]) {
        tc::ld16(tl((isq ? R_Q : R_K) + c0), x);
        rows16(isq ? sInvQ : sInvK, inv);
    };
    // a derived tile, channel-major: bf16(x * m_r * f), m_r = inv_r * mul (hi + lo if lo)
    auto build = [&](unsigned char* tile, unsigned char* lo, bool isq, float mul, int kind) {
        float f[16], x[16], inv[16];
        factors(kind, f);
        load_x(isq, x, inv);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = x[i] * derived_m(inv[i], mul, 1.f) * f[i];
        if (lo)
            store_cm_pair(tile, lo, x);
        else
            store_cm(tile, x);
    };
    // several derived tiles of k at once (e^{gc-ref} and the k rows read from tensor memory
    // once): kd' (e), ki' (1 / e) and, if given, kr (e^{gT-ref} / e); each value exactly as
    // build() forms it.  With `pair`, kd' and ki' are stored as bf16 pairs (lo tiles given).
    auto build_k = [&](unsigned char* kdp, unsigned char* kdp_lo, unsigned char* kip, unsigned char* kip_lo,
                       unsigned char* kr) {
        float e[16], x[16], inv[16], v[16];
        tc::ld16(tl(R_G + c0), e);
        load_x(false, x, inv);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = x[i] * derived_m(inv[i], 1.f, 1.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = x[i] * e[i];
        if (kdp_lo) store_cm_pair(kdp, kdp_lo, v);
        else store_cm(kdp, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = x[i] * __fdividef(1.f, e[i]);
        if (kip_lo) store_cm_pair(kip, kip_lo, v);
        else store_cm(kip, v);
        if (kr) {
            const float eGTref = sFac[MD + L];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = x[i] * __fdividef(eGTref, e[i]);
            store_cm(kr, v);
        }
    };

    // kd (e^{ref} e) and kr (e^{gT-ref} / e) of k at once, each value exactly as build() forms it
    auto build_kr_kd = [&](unsigned char* kr, unsigned char* kd) {
        float e[16], x[16], inv[16], v[16];
        tc::ld16(tl(R_G + c0), e);
        load_x(false, x, inv);
        const float eRef = sFac[L], eGTref = sFac[MD + L];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = x[i] * derived_m(inv[i], 1.f, 1.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = x[i] * (e[i] * eRef);
        store_cm(kd, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = x[i] * __fdividef(eGTref, e[i]);
        store_cm(kr, v);
    };

    // per-thread accumulators (channel L, rows c0 .. c0+15)
    float dQn[NCOL], dKn[NCOL], dGc[NCOL], v[NCOL];
#pragma unroll
    for (int i = 0; i < NCOL; ++i) dQn[i] = dKn[i] = dGc[i] = 0.f;
    // byte offset of element (row c0 + i, column L) in a token-major SW128 tile with `rows` rows
    const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
    auto tok = [&](int rows, int i) -> uint32_t {
        return (uint32_t)((L >> 6) * rows * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
    };

    // ---- G2: X^T = S0^T kd^T, G3: dqd^T = S0 dO^T, G5b: du^T = dS^T kr^T (+ dO^T P later) ----
    // ([A_raw; P] of G1 come from the prep kernel, which computes them for the inverse)
    // kr -> K (the k tile is dead: q and k are staged in tensor memory), kd -> W0 (the raw
    // gate tile is dead after the scan)
    build_kr_kd(sK, sW0);
    sync_all();
    if (tid == 0) {
        constexpr uint32_t id2 = tc::idesc(128, 64, 0, 1), id3 = tc::idesc(128, 64, 1, 0),
                           id5 = tc::idesc(128, 64, 0, 1);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_C, tc::kdesc(sb + oS0, 128, 0, k), tc::mdesc(sb + oW0, 128, 0, k), id2, k > 0);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_D, tc::mdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oDOY, 128, 0, k), id3, k > 0);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_A, tc::kdesc(sb + oDS, 128, 0, k), tc::mdesc(sb + oK, 128, 0, k), id5, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_C + c0), v);
    {
        float bt[16];
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // beta E = beta (V - X), in place of V (lane = value channel)
            __nv_bfloat16* pv = reinterpret_cast<__nv_bfloat16*>(sV + tok(64, i));
            const float be = bt[i] * (__bfloat162float(*pv) - v[i]);
            const __nv_bfloat16 hi = __float2bfloat16(be);
            *pv = hi;
            *reinterpret_cast<__nv_bfloat16*>(sK + tok(64, i)) = __float2bfloat16(be - __bfloat162float(hi));
        }
    }
    tc::ld16(tl(R_D + c0), v);
    {
        float f[16], x[16], inv[16];
        factors(F_KD, f);
        load_x(true, x, inv);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dqd (lane = key channel)
            const float t = p.scale * v[i] * f[i];
            dQn[i] += t;
            dGc[i] += x[i] * inv[i] * t;
        }
    }
    sync_all();

    {  // the item's A and P pair have landed (G5a reads P; the dP / dA epilogue reads A)
        const bool ok = tc::mbar_wait(mAP, (uint32_t)(it & 1));
        if (__syncthreads_or(!ok)) return bail();
        pending_ap = false;
    }
    // ---- G4: u^T = (beta E)^T T^T ; G5a: du^T += dO^T P ------------------------------
    if (tid == 0) {
        constexpr uint32_t id4 = tc::idesc(128, 64, 1, 0), id5 = tc::idesc(128, 64, 1, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oV, 64, 0, k), tc::kdesc(sb + oT, 64, 0, k), id4, k > 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)  // + (beta E lo)^T T^T
            tc::mma(tmem + R_B, tc::mdesc(sb + oK, 64, 0, k), tc::kdesc(sb + oT, 64, 0, k), id4, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_A, tc::mdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oP, 64, 0, k), id5, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)  // + dO^T P lo
            tc::mma(tmem + R_A, tc::mdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oPL, 64, 0, k), id5, 1);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_B + c0), v);
    store_cm_pair(sW1, sW0, v);  // u^T (hi) and its residual (kd is dead)
    tc::ld16(tl(R_A + c0), v);
    store_cm(sW2, v);  // du^T over ki'
    sync_all();

    // ---- G6: dY^T = du^T T ------------------------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id6 = tc::idesc(128, 64, 0, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oW2, 128, 0, k), tc::mdesc(sb + oT, 64, 0, k), id6, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_D + c0), v);
    {
        float bt[16];
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {
            *reinterpret_cast<__nv_bfloat16*>(sW2 + tok(64, i)) = __float2bfloat16(bt[i] * v[i]);  // dv, staged
            *reinterpret_cast<__nv_bfloat16*>(sDOY + tok(128, i) + 64 * 128) = __float2bfloat16(v[i]);  // dY
        }
    }
    sync_all();
    put_tile(&m.dv, true, oW2, 8192, p.dv, ci, h);

    // ---- G7: Z^T = S0 dY^T ; G8: dkr^T = dS u^T ; G9: [dP; dA]_raw = [dO; dY] u^T ------------
    if (tid == 0) {
        constexpr uint32_t id7 = tc::idesc(128, 64, 1, 0), id8 = tc::idesc(128, 64, 1, 1),
                           id9 = tc::idesc(128, 64, 0, 1);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_B, tc::mdesc(sb + oS0, 128, 0, k), tc::kdesc(sb + oDOY, 128, 64, k), id7, k > 0);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_C, tc::mdesc(sb + oDS, 128, 0, k), tc::mdesc(sb + oW1, 128, 0, k), id8, k > 0);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oW1, 128, 0, k), id9, k > 0);
  // u lo
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_C, tc::mdesc(sb + oDS, 128, 0, k), tc::mdesc(sb + oW0, 128, 0, k), id8, 1);
#pragma unroll
        for (int k = 0; k < MD; k += 16)
            tc::mma(tmem + R_D, tc::kdesc(sb + oDOY, 128, 0, k), tc::mdesc(sb + oW0, 128, 0, k), id9, 1);
    
        tc::commit(mb);
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
            const uint4 l = *reinterpret_cast<const uint4*>(sK + tc::sw_chunk(r, j, 64));  // beta E lo
            const uint32_t wl[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = unpack_bf16(wa[e]);
                float2 fb = unpack_bf16(wb[e]);
                const float2 fl = unpack_bf16(wl[e]);
                fb.x += fl.x;
                fb.y += fl.y;
                s2 += fa.x * fb.x + fa.y * fb.y;
            }
        }
        s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
        s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
        if (part == 0) sDbP[r] = s2;
    }
    if (!wait_mma()) return;
    tc::ld16(tl(R_B + c0), v);
    {
        float f[16], x[16], inv[16];
        factors(F_KD, f);
        load_x(false, x, inv);
        float bt[16];
        rows16(sBeta, bt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dkd (from E) = -beta Z
            const float t = -bt[i] * v[i] * f[i];
            dKn[i] += t;
            dGc[i] += x[i] * inv[i] * t;
        }
        tc::ld16(tl(R_C + c0), v);
        factors(F_KR, f);
        float dgt = 0.f;
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dkr
            const float t = v[i] * f[i];
            dKn[i] += t;
            const float kt = x[i] * inv[i] * t;
            dGc[i] -= kt;
            dgt += kt;
        }
        sDgTp[hc * MD + L] = dgt;
    }
    tc::ld16(tl(R_D + c0), v);
    {
        // lanes 0..63: dP rows, lanes 64..127: dA rows ; [dP; beta dA] -> the dS space [128][64]
        const bool isP = L < 64;
        const int r = isP ? L : L - 64;
        const float br = sBeta[r];
        float dbs = 0.f;
        float o[16];
#pragma unroll
        for (int jc = 0; jc < NCOL / 8; ++jc) {
            const uint4 av = *reinterpret_cast<const uint4*>(sA + tc::sw_chunk(r, (c0 >> 3) + jc, 64));
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
                    const float2 aa = unpack_bf16(wa[e]);
                    dbs += a0 * aa.x + a1 * aa.y;
                    a0 *= br;
                    a1 *= br;
                }
                o[i0] = a0;
                o[i0 + 1] = a1;
            }
        }
        if (!isP) sDbA[hc * CH + r] = dbs;
        if (tid == STORE_TID) tc::bulk_wait_read();  // dv's tile is read before qd' takes its space
        __syncthreads();  // every reader of S0, dS (and the u lo tile) is done
        store_cm_pair(sDS, sDS + TILE, o);
    }
    // rebuilds for G10 / G11: ki' -> W0 (lo W1), qd' -> W2 (lo K), kd' -> S0 (lo S0 + 16 KB)
    build_k(sS0, sS0 + TILE, sW0, sW1, nullptr);
    build(sW2, sK, true, p.scale, F_KDP);
    sync_all();
  // the raw gates again, for the gate chain rule, into the dead A and P tiles
    if (tid == 0) {
        tc::mbar_expect_tx(mgr, TILE);
        tc::tma_load_4d(sb + oA, &m.graw, 0, h, (int)ci.t0, 0, mgr);
    }
    pending_g = true;

    // ---- G10: [dqd', dkd']^T = ki'^T [dP; beta dA]^T ; G11: dki'^T = qd'^T dP + kd'^T (beta dA) --
    if (tid == 0) {
        constexpr uint32_t id10 = tc::idesc(128, 128, 0, 0), id11 = tc::idesc(128, 64, 0, 1);
        const uint32_t kiH = sb + oW0, kiL = sb + oW1, qdH = sb + oW2, qdL = sb + oK, kdH = sb + oS0,
                       kdL = sb + oS0 + TILE, xH = sb + oDS, xL = sb + oDS + TILE;
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_A, tc::kdesc(kiH, 128, 0, k), tc::kdesc(xH, 128, 0, k), id10, k > 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_A, tc::kdesc(kiH, 128, 0, k), tc::kdesc(xL, 128, 0, k), id10, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_A, tc::kdesc(kiL, 128, 0, k), tc::kdesc(xH, 128, 0, k), id10, 1);
    
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::kdesc(qdH, 128, 0, k), tc::mdesc(xH, 128, 0, k), id11, k > 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_B, tc::kdesc(kdH, 128, 0, k), tc::mdesc(xH, 128, 64, k), id11, 1);
#pragma unroll
        for (int k = 0; k < CH; k += 16) {
            tc::mma(tmem + R_B, tc::kdesc(qdH, 128, 0, k), tc::mdesc(xL, 128, 0, k), id11, 1);
            tc::mma(tmem + R_B, tc::kdesc(qdL, 128, 0, k), tc::mdesc(xH, 128, 0, k), id11, 1);
            tc::mma(tmem + R_B, tc::kdesc(kdH, 128, 0, k), tc::mdesc(xL, 128, 64, k), id11, 1);
            tc::mma(tmem + R_B, tc::kdesc(kdL, 128, 0, k), tc::mdesc(xH, 128, 64, k), id11, 1);
        }
    
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    // every large shared tile is dead: the next item's operands may land while this epilogue runs
    if (item + (int)gridDim.x < n_items) {
        const ChunkInfo cn = get_ci((it + 1) & 1);
        if (lane == 0 && warp < 9) issue_loads(item + gridDim.x, cn, warp);  // one copy per warp
        pending = true;
        pend_par = (uint32_t)((it + 1) & 1);
        prefetch_small(item + gridDim.x, cn);
    }
    // the gate-gradient term takes the derived-tile value the products consumed: the fp32
    // value of the hi + lo pair
    auto tile_val = [&](float x, float mm, float f) -> float { return x * mm * f; };
    {
        float f[16], x[16], inv[16];
        factors(F_KDP, f);
        load_x(true, x, inv);
        tc::ld16(tl(R_A + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dqd'
            dQn[i] += p.scale * v[i] * f[i];
            dGc[i] += tile_val(x[i], derived_m(inv[i], p.scale, 1.f), f[i]) * v[i];
        }
        load_x(false, x, inv);
        tc::ld16(tl(R_A + 64 + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dkd'
            dKn[i] += v[i] * f[i];
            dGc[i] += tile_val(x[i], derived_m(inv[i], 1.f, 1.f), f[i]) * v[i];
        }
        factors(F_KIP, f);
        tc::ld16(tl(R_B + c0), v);
#pragma unroll
        for (int i = 0; i < NCOL; ++i) {  // dki'
            dKn[i] += v[i] * f[i];
            dGc[i] -= tile_val(x[i], derived_m(inv[i], 1.f, 1.f), f[i]) * v[i];
        }
    }

    // ---- epilogue: L2-norm backward, dq / dk, dbeta, the gate gradient ----------------------
    float* sRowQ = sRow;        // [4][64] per lane quarter
    float* sRowK = sRow + 256;  // [4][64]
    {
        // per-row dots over this warp's 32 channels: lane l gets row c0 + (l & 15)
        float t[32];
        {
            float x[16], inv[16];
            load_x(true, x, inv);
#pragma unroll
            for (int i = 0; i < NCOL; ++i) t[i] = dQn[i] * x[i] * inv[i];
            load_x(false, x, inv);
#pragma unroll
            for (int i = 0; i < NCOL; ++i) t[16 + i] = dKn[i] * x[i] * inv[i];
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
        float x[16], inv[16], tt[16];
        load_x(true, x, inv);
        rows16(sTot, tt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i)  // dq into the dead ki' lo tile
            *reinterpret_cast<__nv_bfloat16*>(sW1 + tok(64, i)) =
                __float2bfloat16((dQn[i] - x[i] * inv[i] * tt[i]) * inv[i]);
        load_x(false, x, inv);
        rows16(sTot + CH, tt);
#pragma unroll
        for (int i = 0; i < NCOL; ++i)  // dk into the dead dY rows (the next item's dO fills rows 0..63)
            *reinterpret_cast<__nv_bfloat16*>(sDOY + tok(128, i) + 64 * 128) =
                __float2bfloat16((dKn[i] - x[i] * inv[i] * tt[i]) * inv[i]);
    }
    sync_all();
    put_tile(&m.dq, true, oW1, 8192, p.dq, ci, h);
    put_tile(&m.dk, false, oDOY + 64 * 128, 128 * 128, p.dk, ci, h);
    // dbeta (logit space)
    for (int r = tid; r < ci.len; r += 512) {
        const float dA_A = ((sDbA[r] + sDbA[CH + r]) + sDbA[2 * CH + r]) + sDbA[3 * CH + r];
        p.dbeta[(ci.t0 + r) * p.H + h] = __float2bfloat16(sBeta[CH + r] * (sDbP[r] + dA_A));
    }
    auto dgT_of = [&](int d) -> float {
        return (((sDgTs[d] + sDgTp[d]) + sDgTp[MD + d]) + sDgTp[2 * MD + d]) + sDgTp[3 * MD + d];
    };
    // reverse cumsum of dgc over the rows per channel: this thread's 16 rows in registers,
    // the later row quarters' totals and the chunk constant dgT as the suffix; then the
    // gate chain rule per element, with per-channel partial sums
    float sfx = 0.f;
#pragma unroll
    for (int i = 15; i >= 0; --i) {
        sfx += dGc[i];
        dGc[i] = sfx;
    }
    sScan[hc * MD + L] = sfx;  // read after the barrier of the raw-gate wait below
    float xr[16];
    const float dtb = sGate[L];
    {
        const bool ok = tc::mbar_wait(mgr, (uint32_t)(it & 1));
        if (__syncthreads_or(!ok)) return bail();
        pending_g = false;
        const unsigned char* gt = smem + oA;  // token-major raw gates (A and P spaces)
        const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
            xr[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(gt + off)) + dtb;
        }
    }
    float post = dgT_of(L);
#pragma unroll
    for (int h2 = 3; h2 >= 0; --h2)
        if (h2 > hc) post += sScan[h2 * MD + L];
    const float ea = sMisc[32];
    float ddt = 0.f, dA_acc = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = c0 + i;
        float dA;
        const float draw = kda_gate_bwd<GATE>(p.gate_scale, ea, xr[i], dGc[i] + post, dA);
        // staged in the raw-gate tile (read into xr above); rows past the end add nothing
        *reinterpret_cast<__nv_bfloat16*>(smem + oA + tok(64, i)) = __float2bfloat16(draw);
        if (r < ci.len) {
            ddt += draw;
            dA_acc += dA;
        }
    }
    // the partial sums go to the row-dot space (dead since the L2 backward) and the
    // per-warp slots, so that one barrier serves them and the staged dg_raw
    sRow[hc * MD + L] = ddt;
    dA_acc = warp_sum(dA_acc);
    if (lane == 0) sMisc[warp] = dA_acc;
    sync_all();  // dg_raw staged; partial sums written
    put_tile(&m.dgr, true, oA, 8192, p.dg_raw, ci, h);
    if (tid < MD) {
        const float t = ((sRow[tid] + sRow[MD + tid]) + sRow[2 * MD + tid]) + sRow[3 * MD + tid];
        atomicAdd(&p.ddt_bias[h * MD + tid], t);
    }
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < 16; ++w) t += sMisc[w];
        atomicAdd(&p.dA_log[h], t);
    }
    tc::fence_before();
    __syncthreads();  // this item's small arrays and tensor memory are free
    tc::fence_after();
    }
    if (tid == STORE_TID) tc::bulk_wait_all();
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

template <int GATE>
static cudaError_t launch_main_kda_t(const Params& p, cudaStream_t s) {
    MainMaps m;
    const uint64_t rows_cc = (uint64_t)p.max_chunks * p.H * CH;
    const uint64_t rows_dd = (uint64_t)p.max_chunks * p.H * MD;
    const uint64_t T = (uint64_t)p.T_total;
    bool ok = encode_blocked_tokens_map(&m.q, p.q, T, p.Hk) && encode_blocked_tokens_map(&m.k, p.k, T, p.Hk) &&
              encode_blocked_tokens_map(&m.v, p.v, T, p.H) && encode_tokens_map(&m.dO, p.dO, T, p.H, MD) &&
              encode_blocked_rows_map(&m.S0, p.S0, rows_dd, MD) && encode_blocked_rows_map(&m.dS, p.dS, rows_dd, MD) &&
              encode_rows_map(&m.T, p.Tm, rows_cc, CH, CH) && encode_rows_map(&m.ap, p.APm, 3 * rows_cc, CH, CH) &&
              encode_blocked_tokens_map(&m.graw, p.g_raw, T, p.H) &&
              encode_blocked_tokens_map(&m.dq, p.dq, T, p.H) && encode_tokens_map(&m.dk, p.dk, T, p.H, MD) &&
              encode_blocked_tokens_map(&m.dv, p.dv, T, p.H) &&
              encode_blocked_tokens_map(&m.dgr, p.dg_raw, T, p.H);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_main_kda<GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int items = p.max_chunks * p.H;
    const int ctas = items < num_sms() ? items : num_sms();
    k_main_kda<GATE><<<ctas, 512, SMEM_BYTES, s>>>(p, m);
    return cudaGetLastError();
}

cudaError_t launch_main_kda(const Params& p, cudaStream_t s) {
    // the KDA gate function is a template parameter: each instance carries only its own code
    return p.kda_gate == 0 ? launch_main_kda_t<0>(p, s) : launch_main_kda_t<1>(p, s);
}

}  // namespace gdr
