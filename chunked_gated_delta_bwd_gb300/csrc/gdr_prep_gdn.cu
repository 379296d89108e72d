// Chunk-parallel preparation on tcgen05 for D = 128 with the scalar (GDN) gate:
// persistent CTAs of 16 warps, one per SM, each looping over (chunk, head) items, with two
// input stages.  The quantities of the X/R form of the FlashQLA dh kernel ("FlashQLA ...
// GDN 反向", §三), as the per-channel kernel in gdr_prep_kda.cu computes them:
//
//   [A; P] = [kd'; qd'] ki'^T        A = strict_lower(diag(beta) .) (fp32), P = lower(.)
//   T   = (I + A)^-1                  W^T = (beta kd)^T T^T       U^T = (beta V)^T T^T
//   R^T = qd^T - W^T P^T (a bf16 pair R_hi + R_lo)                kr  = kn e^{gT-gc}
//
// With one log gate per token every gated tile is a row scaling of the raw q or k tile,
// so, as in the scalar-gate main kernel, the products read the raw bf16 tiles as loaded
// (k and q stacked into one 128-row tile) and the row factors are applied in fp32:
//   G1  [A; P]_raw = [k; q] k^T, then A = G1 x beta_r invk_r e^{gc_r-ref} x invk_s e^{ref-gc_s}
//       and P = G1 x scale invq_r e^{gc_r-ref} x invk_s e^{ref-gc_s};
//   W^T = k^T (T diag(beta invk e^{gc}))^T and U^T = v^T (T diag(beta))^T: the column
//       factors go into two bf16 copies of T, no (beta kd)^T or (beta V)^T tile is built.
//
// Schedule of one item: the row norms, gate factors and combined row factors (all warps);
// E1 (A, P) from G1; then warps 0..7 invert T while warps 8..15 build kr and run the NEXT
// item's front part (the wait for its tiles, its raw q, k rows into tensor memory, its G1
// issued on the raw tiles) and warps 6, 7 (free after the inverse's diagonal blocks) scan the
// next item's gates and beta and look up the chunk of the item after it (small arrays and
// those tensor-memory columns are kept per item parity); then T1, T2, the W / U product, R.  A stage's tiles are last
// read by the W / U product, after which the tiles of the item after next are loaded into it.
// W, U, Kr, R_hi, R_lo and T are staged in shared tiles that are dead by then (none in an
// input stage) and written by TMA stores that one thread issues.
#include "gdr_chunk.cuh"
#include "gdr_invert.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"

namespace gdr {

namespace {

using inv::LDF;
using inv::XLD;
constexpr int PD = 128;
constexpr int TILE = CH * PD * 2;  // 16 KB
// shared-memory map (bytes from the 1024-aligned base); two input stages
constexpr int STAGE = 3 * TILE;
constexpr int oKQ = 0;            // [k; q] token-major, 128 rows
constexpr int oV = 2 * TILE;      // v token-major
constexpr int oW2 = 2 * STAGE;    // kr staged [d][r] -> W^T bf16 [d][s] (R's operand, W's store)
constexpr int oP = oW2 + TILE;    // P [r][s] bf16
constexpr int oT = oP + 8192;     // T [r][s] bf16 (blocks above the diagonal stay zero)
constexpr int oT1 = oT + 8192;    // T diag(beta invk e^{gc}) [r][s] bf16 -> (with T2's space) R_lo^T staged
constexpr int oT2 = oT1 + 8192;   // T diag(beta) [r][s] bf16
constexpr int oA = oT2 + 8192;    // A fp32 [64][LDF] row-major -> U^T staged [j][s]
static_assert(oA % 1024 == 0, "U's staging tile is 128-byte swizzled");
constexpr int oTf = oA + CH * LDF * 4;    // T fp32, transposed [c][r], stride LDF -> R_hi^T staged [d][r]
static_assert(oTf % 1024 == 0, "R_hi's staging tile is 128-byte swizzled");
constexpr int oTmp = oTf + CH * LDF * 4;  // 8 warps' transfer tiles [8][XLD]
constexpr int nTmp = 8 * 8 * XLD;
constexpr int oSmall = (oTmp + nTmp * 4 + 1023) / 1024 * 1024;
// one set per item parity (an item's front part fills its set while the item before it is
// still in flight): inverse norms of q and k, beta, gate factors, gates gc[64], ref, gT
constexpr int nInvQ = 64, nInvK = 64, nBeta = 64, nFac = 4 * 64, nGate = 68;
constexpr int nPar = nInvQ + nInvK + nBeta + nFac + nGate;
constexpr int nTab = 4 * 64, nPad = 8;
constexpr int SMALL_FLOATS = 2 * nPar + nTab + nPad;
constexpr int SMEM_BYTES = oSmall + SMALL_FLOATS * 4 + 128 + 1024;  // + barriers, tensor-memory slot, chunk info
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(nPar % 4 == 0, "16-byte aligned per-parity arrays");
// tensor-memory columns; raw q, k rows of item parity x at R_Q0 + 128 x, R_K0 + 128 x
constexpr uint32_t R_G1 = 0, R_W = 64, R_U = 128, R_R = 192, R_Q0 = 256, R_K0 = 320;
// combined row-factor tables (each [64])
enum Tab { T_CF = 0, T_RA = 1, T_RP = 2, T_CW = 3 };
// The thread that issues the TMA stores of W, U, Kr, R_hi, R_lo and T (a bulk store's
// completion is visible only to the thread that issued it, so it also waits for their reads
// of the staging tiles before those are rewritten) and the q, k, v copies (a warp 8..15
// thread, so that the next item's front clears its record of a copy in flight).
constexpr int STORE_TID = 416;

struct PrepGdnMaps {
    CUtensorMap q, k, v, W, U, Kr, R, Rlo, T;
};

}  // namespace

__global__ void __launch_bounds__(512, 1) k_prep_gdn(const Params p, const __grid_constant__ PrepGdnMaps m) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // items (chunk, head) = chunk * H + h over the chunks that exist
    const int total_chunks = p.chunk_off ? p.chunk_off[p.N] : p.N * (int)((p.seq_len + CH - 1) / CH);
    const int n_items = total_chunks * p.H;
    const int q4 = warp & 3, hc = warp >> 2;
    const int L = 32 * q4 + lane;  // this thread's lane: a channel, or a stacked row of G1
    const int c0 = 16 * hc;        // first of this thread's 16 rows (or columns)

    unsigned char *sW2 = smem + oW2, *sP = smem + oP, *sT = smem + oT, *sT1 = smem + oT1, *sT2 = smem + oT2;
    float* sA = reinterpret_cast<float*>(smem + oA);
    float* sTf = reinterpret_cast<float*>(smem + oTf);
    float* sTmp = reinterpret_cast<float*>(smem + oTmp);
    float* fsm = reinterpret_cast<float*>(smem + oSmall);
    // per-parity small arrays of the item with parity x
    auto sInvQ = [&](int x) { return fsm + x * nPar; };
    auto sInvK = [&](int x) { return fsm + x * nPar + nInvQ; };
    auto sBeta = [&](int x) { return fsm + x * nPar + nInvQ + nInvK; };
    auto sFac = [&](int x) {  // [4][64] e^{gc}, e^{gc-ref}, e^{ref-gc}, e^{gT-gc} (Fac order)
        return fsm + x * nPar + nInvQ + nInvK + nBeta;
    };
    auto gates = [&](int x) {
        ScalarGates G;
        G.gc = fsm + x * nPar + nInvQ + nInvK + nBeta + nFac;
        G.ref = G.gc + CH;
        G.gT = G.gc + CH + 1;
        return G;
    };
    float* sTab = fsm + 2 * nPar;  // [4][64] combined row factors of the current item (Tab order)
    uint64_t* mbars = reinterpret_cast<uint64_t*>(sTab + nTab + nPad);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbars + 4);
    // chunk info of the items of parity 0 and 1 (an item's slot is filled two items ahead: the
    // lookup's dependent integer chain costs hundreds of cycles inside the busy loop)
    int* sCI = reinterpret_cast<int*>(mbars + 6);
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
    // product barrier, load barriers (one per stage), G1 barrier
    const uint32_t mb = smem_u32(mbars), mload0 = smem_u32(mbars + 1), mg1 = smem_u32(mbars + 3);

    // q, k, v of `item` into stage `stg`: k and q stacked into one 128-row tile, one 64-column
    // box at a time, v as two column blocks; copy `which` (0..4; the barrier's byte count goes
    // with copy 4), or all five for which < 0
    auto issue_loads = [&](int item, const ChunkInfo& cj, int stg, int which) {
        const int hh = item % p.H, hk = qk_head(p, hh), t0 = (int)cj.t0;
        const uint32_t bar = mload0 + 8 * stg, st = sb + stg * STAGE;
        if (which < 0 || which == 4) tc::mbar_expect_tx(bar, 3 * TILE);
        if (which < 0 || which == 0) tc::tma_load_3d(st + oKQ, &m.k, 0, hk, t0, bar);
        if (which < 0 || which == 1) tc::tma_load_3d(st + oKQ + 2 * 8192, &m.k, 64, hk, t0, bar);
        if (which < 0 || which == 2) tc::tma_load_3d(st + oKQ + 8192, &m.q, 0, hk, t0, bar);
        if (which < 0 || which == 3) tc::tma_load_3d(st + oKQ + 3 * 8192, &m.q, 64, hk, t0, bar);
        if (which < 0 || which == 4) tc::tma_load_4d(st + oV, &m.v, 0, hh, t0, 0, bar);
    };
    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) {
        tc::mbar_init(mb, 1);
        tc::mbar_init(mload0, 1);
        tc::mbar_init(mload0 + 8, 1);
        tc::mbar_init(mg1, 1);
        for (int j = 0; j < 2; ++j) {  // the first two items' chunk info
            ChunkInfo c{};
            if ((int)blockIdx.x + j * (int)gridDim.x < n_items)
                lookup_chunk(((int)blockIdx.x + j * (int)gridDim.x) / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, c);
            put_ci(j, c);
        }
    }
    // T's blocks above the diagonal stay zero in the shared tile
    for (int i = tid; i < CH * CH * 2 / 16; i += 512)
        *reinterpret_cast<uint4*>(smem + oT + 16 * i) = make_uint4(0, 0, 0, 0);
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // bit j: stage j has a load in flight (the store thread's view) / that load's barrier parity
    uint32_t pend = 0, pend_par = 0;
    if (tid == STORE_TID)
        for (int j = 0; j < 2; ++j)
            if ((int)blockIdx.x + j * (int)gridDim.x < n_items) {
                issue_loads(blockIdx.x + j * gridDim.x, get_ci(j), j, -1);
                pend |= 1u << j;
            }
    const uint32_t tmem = *tslot;
    uint32_t phase = 0;
    int it = 0;  // this CTA's item count (selects the stage and the parity of the small arrays)
    auto tl = [&](uint32_t col) { return tmem + ((uint32_t)(32 * q4) << 16) + col; };
    auto sync_all = [&]() {
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    auto bail = [&]() {
        if (tid == STORE_TID) {
            for (int j = 0; j < 2; ++j)
                if ((pend >> j) & 1) tc::mbar_wait(mload0 + 8 * j, (pend_par >> j) & 1);  // bounded drain
            tc::bulk_wait_all();
        }
        if (tid == 0) atomicOr(p.status, ST_MMA_TIMEOUT);
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
    // An item's gates (warp 6, lane l: rows 2l and 2l + 1) and beta logits (warp 7, lane l:
    // rows l and l + 32), read as raw values (rows clamped into the chunk) a full item before
    // warps 6 and 7, idle once the inversion's diagonal blocks are done, scan them.
    float pg0 = 0.f, pg1 = 0.f;
    unsigned short pb0 = 0, pb1 = 0;
    auto prefetch_small = [&](int item, const ChunkInfo& cj) {
        const int hh = item % p.H;
        if (warp == 6) {
            pg0 = p.g[(cj.t0 + min(2 * lane, cj.len - 1)) * p.H + hh];
            pg1 = p.g[(cj.t0 + min(2 * lane + 1, cj.len - 1)) * p.H + hh];
        } else if (warp == 7) {
            const unsigned short* bl = reinterpret_cast<const unsigned short*>(p.beta_logit);
            pb0 = bl[(cj.t0 + min(lane, cj.len - 1)) * p.H + hh];
            pb1 = bl[(cj.t0 + min(lane + 32, cj.len - 1)) * p.H + hh];
        }
    };
    // warps 6 and 7: gates and beta of the item of parity x (raw values read an item before)
    auto scan_small = [&](int x, const ChunkInfo& cj) {
        if (warp == 6) {
            gdn_gate_scan(2 * lane < cj.len ? pg0 : 0.f, 2 * lane + 1 < cj.len ? pg1 : 0.f, gates(x), true, p);
        } else if (warp == 7) {
            sBeta(x)[lane] = lane < cj.len ? sigmoid_f(__bfloat162float(__ushort_as_bfloat16(pb0))) : 0.f;
            sBeta(x)[lane + 32] = lane + 32 < cj.len ? sigmoid_f(__bfloat162float(__ushort_as_bfloat16(pb1))) : 0.f;
        }
    };
    auto rows16 = [&](const float* a, float (&o)[16], int cq) {  // a[cq .. cq+15]
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = *reinterpret_cast<const float4*>(a + cq + 4 * i);
            o[4 * i] = v.x;
            o[4 * i + 1] = v.y;
            o[4 * i + 2] = v.z;
            o[4 * i + 3] = v.w;
        }
    };
    auto pack8 = [&](const float (&v)[16], uint32_t (&w)[8]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
    };
    // row L, columns cq .. cq+15 of a channel-major [128][64] shared tile
    auto store_cm = [&](unsigned char* tile, const uint32_t (&w)[8], int cq) {
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, cq >> 3, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(tile + tc::sw_chunk(L, (cq >> 3) + 1, 128)) = make_uint4(w[4], w[5], w[6], w[7]);
    };
    // raw q (or k) of this thread's channel and rows cq .. cq+15 (staged in tensor memory for
    // the item of parity x) times the rows' inverse norm, the multiplier and the gate factor
    // `kind`
    auto derived = [&](int x, bool isq, float mul, int kind, float (&o)[16], int cq) {
        float f[16], inv[16];
        rows16(sFac(x) + kind * CH, f, cq);
        tc::ld16(tl((isq ? R_Q0 : R_K0) + 128 * x + cq), o);
        rows16(isq ? sInvQ(x) : sInvK(x), inv, cq);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = o[i] * derived_m(inv[i], mul, 1.f) * f[i];
    };
    // The front part of item number `itx` of this CTA, on warps 8..15 (u = tid - 256): what
    // needs no product of the item before it.  It runs while warps 0..7 invert T of the item
    // before (the first item's runs before the loop): the wait for the item's q, k, v tiles,
    // rows past the chunk's end zeroed, its raw q and k rows into the tensor-memory columns of
    // the item's parity, and G1 = [k; q] k^T issued on the raw tiles (warp 15).  False (on
    // every participant) if the wait for the tiles timed out.
    auto front = [&](int item, int itx) -> bool {
        const int u = tid - 256, x = itx & 1;
        const bool ok = tc::mbar_wait(mload0 + 8 * x, (uint32_t)((itx >> 1) & 1));
        if (tc::named_or(2, 256, !ok)) return false;
        if (tid == STORE_TID) pend &= ~(1u << x);
        const ChunkInfo cf = get_ci(x);
        unsigned char* kq = smem + x * STAGE + oKQ;
        if (cf.len < CH) {
            const int nz = (CH - cf.len) * 16;  // 16-byte chunks per 128-column row
            for (int i = u; i < 3 * nz; i += 256) {
                const int t = i / nz, rem = i % nz, r = cf.len + rem / 16, jc = rem % 16;
                unsigned char* base = t < 2 ? kq : smem + x * STAGE + oV;
                const int row = t == 1 ? 64 + r : r, rows = t == 2 ? 64 : 128;
                *reinterpret_cast<uint4*>(base + tc::sw_chunk(row, jc, rows)) = make_uint4(0, 0, 0, 0);
            }
            tc::fence_async_smem();
            tc::named_sync(2, 256);
        }
        {  // raw q and k of this thread's channel, row blocks hc - 2 and hc, into tensor memory
            const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
            for (int pass = 0; pass < 2; ++pass) {
                const int cb = 16 * (hc - 2 + 2 * pass);
                float qs[16], ks[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {  // k row cb + i; the q row sits 64 rows (8 KB) below
                    const uint32_t off = (uint32_t)((L >> 6) * 128 * 128 + (cb + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
                    ks[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(kq + off));
                    qs[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(kq + off + 64 * 128));
                }
                tc::st16(tl(R_Q0 + 128 * x + cb), qs);
                tc::st16(tl(R_K0 + 128 * x + cb), ks);
            }
        }
        if (u == 224) {  // G1 on the tiles as loaded (by the last warp); the item's E1 waits for it
            constexpr uint32_t id1 = tc::idesc(128, 64, 0, 0);
            const uint32_t a = sb + x * STAGE + oKQ;
#pragma unroll
            for (int k = 0; k < PD; k += 16) tc::mma(tmem + R_G1, tc::kdesc(a, 128, 0, k), tc::kdesc(a, 128, 0, k), id1, k > 0);
            tc::commit(mg1);
        }
        return true;
    };
    {  // the first item's front
        bool fok = true;
        if ((int)blockIdx.x < n_items) {  // (a packed batch can have fewer items than CTAs)
            if (warp == 6 || warp == 7) {  // gates and beta of the first item; raw values of the second
                prefetch_small(blockIdx.x, get_ci(0));
                scan_small(0, get_ci(0));
                if ((int)blockIdx.x + (int)gridDim.x < n_items) prefetch_small(blockIdx.x + gridDim.x, get_ci(1));
            }
            if (tid >= 256) fok = front(blockIdx.x, 0);
        }
        tc::fence_before();
        if (__syncthreads_or(!fok)) return bail();
        tc::fence_after();
    }

    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const int chunk = item / p.H, h = item % p.H;
    const int stg = it & 1, x = stg;  // the stage and the parity of the small arrays
    const uint32_t st = sb + stg * STAGE;
    unsigned char* sKQ = smem + stg * STAGE + oKQ;
    const size_t tile_cc = ((size_t)chunk * p.H + h) * CH * CH;
    const int trow = (chunk * p.H + h) * PD;  // the chunk-head's first row in the [D][C] tile maps
    const bool has_next = item + (int)gridDim.x < n_items;
    // the last item's W, U store has read A's tile (written by E1); its R store (the latest
    // group) is waited for before the inversion
    if (tid == STORE_TID) tc::bulk_wait_read_but1();
    {  // inverse row norms (8 threads per row: 4 for q, 4 for k), the gate factors and the
       // combined row factors of row r, from the front's gates and beta
        // (chunks p + 4i of the q row and p + 4 + 4i of the k row: the 8 threads of a row read
        // 8 different 16-byte bank groups)
        const int r = tid >> 3, part = tid & 7, row = part < 4 ? 64 + r : r;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = ((part & 3) + 4 * i + (part & 4)) & 15;
            const uint4 v = *reinterpret_cast<const uint4*>(sKQ + tc::sw_chunk(row, j, 128));
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16(wv[e]);
                s += f.x * f.x + f.y * f.y;
            }
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        const float sk = __shfl_xor_sync(0xffffffffu, s, 4);
        if (part == 0) {
            const ScalarGates G = gates(x);
            const float iq = rsqrtf(s + 1e-6f), ik = rsqrtf(sk + 1e-6f), bt = sBeta(x)[r];
            const float fkd = gate_factor<F_KD>(G, r), fkdp = gate_factor<F_KDP>(G, r);
            const float fkip = gate_factor<F_KIP>(G, r), fkr = gate_factor<F_KR>(G, r);
            float* fac = sFac(x);
            sInvQ(x)[r] = iq;
            sInvK(x)[r] = ik;
            fac[F_KD * CH + r] = fkd;
            fac[F_KDP * CH + r] = fkdp;
            fac[F_KIP * CH + r] = fkip;
            fac[F_KR * CH + r] = fkr;
            sTab[T_CF * CH + r] = ik * fkip;          // ki' column factor
            sTab[T_RA * CH + r] = bt * ik * fkdp;     // A row factor (with beta)
            sTab[T_RP * CH + r] = p.scale * iq * fkdp;  // P row factor
            sTab[T_CW * CH + r] = bt * ik * fkd;      // column factor of T for W
        }
    }
    {  // G1, issued by the front (its barrier also publishes the tables)
        const bool ok = tc::mbar_wait(mg1, (uint32_t)(it & 1));
        tc::fence_after();
        if (__syncthreads_or(!ok)) return bail();
    }
    {
        float v[16], cf[16];
        tc::ld16(tl(R_G1 + c0), v);
        rows16(sTab + T_CF * CH, cf, c0);
        if (L < 64) {  // A = strict_lower(beta A_raw), fp32 for the inversion
            const int r = L;
            const float rf = sTab[T_RA * CH + r];
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(sA + r * LDF + c0 + i) =
                    make_float4(c0 + i < r ? v[i] * rf * cf[i] : 0.f, c0 + i + 1 < r ? v[i + 1] * rf * cf[i + 1] : 0.f,
                                c0 + i + 2 < r ? v[i + 2] * rf * cf[i + 2] : 0.f,
                                c0 + i + 3 < r ? v[i + 3] * rf * cf[i + 3] : 0.f);
        } else {  // P = lower(qd' ki'^T), bf16 [r][s]
            const int r = L - 64;
            const float rf = sTab[T_RP * CH + r];
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s0 = c0 + 2 * e;
                w[e] = pack_bf16(s0 <= r ? v[2 * e] * rf * cf[2 * e] : 0.f,
                                 s0 + 1 <= r ? v[2 * e + 1] * rf * cf[2 * e + 1] : 0.f);
            }
            *reinterpret_cast<uint4*>(sP + tc::sw_chunk(r, c0 >> 3, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(sP + tc::sw_chunk(r, (c0 >> 3) + 1, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
            if (p.Pm) {  // forward output: P [r][s] per chunk-head
                uint4* g = reinterpret_cast<uint4*>(p.Pm + tile_cc + r * CH + c0);
                g[0] = make_uint4(w[0], w[1], w[2], w[3]);
                g[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
    if (tid == STORE_TID) tc::bulk_wait_read();  // the last item's R stores have read T's fp32 tile and T1
    sync_all();  // A and P staged; G1's tensor memory has been read (the next item's G1 reuses it)
    bool fok = true;
    if (warp < 8) {
        inv::invert_tc(sA, sTf, sTmp, sT, nullptr);
        if (warp >= 6) {  // (warps 6, 7 leave the inversion after its diagonal blocks)
            // the next item's gates and beta; the chunk info of the item after it (into this
            // item's slot) and its raw gates and beta
            if (has_next) scan_small(x ^ 1, get_ci(x ^ 1));
            if (item + 2 * (int)gridDim.x < n_items) {
                ChunkInfo c2;
                lookup_chunk((item + 2 * (int)gridDim.x) / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, c2);
                if (tid == 192) put_ci(x, c2);
                prefetch_small(item + 2 * gridDim.x, c2);
            }
        }
    } else {
        // meanwhile: kr = kn e^{gT-gc} (this warp's lanes, row quarters hc - 2 and hc) into the
        // W^T tile, which W's epilogue fills only after kr's store has read it; gT, e^{gT}; then
        // the next item's front
        uint32_t w[8];
        for (int pass = 0; pass < 2; ++pass) {
            const int cq = 16 * (hc - 2 + 2 * pass);
            float v[16];
            derived(x, false, 1.f, F_KR, v, cq);
            pack8(v, w);
            store_cm(sW2, w, cq);
        }
        tc::fence_async_smem();
        if (hc == 2) {
            const float gt = gates(x).gTv();
            p.gT[((size_t)chunk * p.H + h) * PD + L] = gt;
            p.egT[((size_t)chunk * p.H + h) * PD + L] = __expf(gt);
        }
        if (has_next) fok = front(item + gridDim.x, it + 1);
    }
    // T complete (fp32 transposed in sTf, bf16 in sT); kr staged; the next item's front done
    tc::fence_before();
    if (__syncthreads_or(!fok)) return bail();
    tc::fence_after();
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.Kr, 0, trow, sb + oW2);
        tc::bulk_commit();
    }
    {
        // T diag(beta invk e^{gc}) -> T1 and T diag(beta) -> T2 (bf16 [r][s]), the B operands of
        // W^T = k^T T1^T and U^T = v^T T2^T; thread: row r, 16 columns, one of the two copies
        const int r = tid & 63, cq = 16 * ((tid >> 6) & 3), which = tid >> 8;
        float f[16];
        rows16(which == 0 ? sTab + T_CW * CH : sBeta(x), f, cq);
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = cq + i <= r ? sTf[(cq + i) * LDF + r] * f[i] : 0.f;
        uint32_t w[8];
        pack8(v, w);
        unsigned char* dst = which == 0 ? sT1 : sT2;
        *reinterpret_cast<uint4*>(dst + tc::sw_chunk(r, cq >> 3, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + tc::sw_chunk(r, (cq >> 3) + 1, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    sync_all();
    if (tid == STORE_TID) {  // T for the main backward
        tc::tma_store_2d(&m.T, 0, (chunk * p.H + h) * CH, sb + oT);
        tc::bulk_commit();
    }

    // ---- W^T = k^T T1^T ; U^T = v^T T2^T ------------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 1, 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_W, tc::mdesc(st + oKQ, 128, 0, k), tc::kdesc(sb + oT1, 64, 0, k), id, k > 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_U, tc::mdesc(st + oV, 64, 0, k), tc::kdesc(sb + oT2, 64, 0, k), id, k > 0);
        tc::commit(mb);
    }
    if (tid == STORE_TID) tc::bulk_wait_read();  // kr's store has read the W^T tile
    if (!wait_mma()) return;
    // the products have read this stage for the last time: the tiles of the item after next
    // go into it, more than an item ahead of that item's front
    if (tid == STORE_TID && item + 2 * (int)gridDim.x < n_items) {
        issue_loads(item + 2 * gridDim.x, get_ci(x), stg, -1);
        pend |= 1u << stg;
        pend_par = (pend_par & ~(1u << stg)) | ((uint32_t)(((it + 2) >> 1) & 1) << stg);
    }
    {
        float v[16];
        uint32_t w[8];
        tc::ld16(tl(R_W + c0), v);
        pack8(v, w);
        store_cm(sW2, w, c0);  // bf16 W^T [d][s]: the A operand of W^T P^T and W's store
        tc::ld16(tl(R_U + c0), v);
        pack8(v, w);
        store_cm(reinterpret_cast<unsigned char*>(sA), w, c0);  // U^T over the dead fp32 A
    }
    sync_all();
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.W, 0, trow, sb + oW2);
        tc::tma_store_2d(&m.U, 0, trow, sb + oA);
        tc::bulk_commit();
    }

    // ---- R^T = qd^T - W^T P^T ----------------------------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 0, 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_R, tc::kdesc(sb + oW2, 128, 0, k), tc::kdesc(sb + oP, 64, 0, k), id, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    {
        float acc[16], qd[16];
        uint32_t w[8], wl[8];
        tc::ld16(tl(R_R + c0), acc);
        derived(x, true, p.scale, F_KD, qd, c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float r0 = qd[2 * e] - acc[2 * e], r1 = qd[2 * e + 1] - acc[2 * e + 1];
            w[e] = pack_bf16(r0, r1);
            const float2 hf = unpack_bf16(w[e]);
            wl[e] = pack_bf16(r0 - hf.x, r1 - hf.y);
        }
        store_cm(reinterpret_cast<unsigned char*>(sTf), w, c0);  // R_hi over the dead fp32 T
        store_cm(sT1, wl, c0);        // R_lo over the dead T1, T2
        tc::fence_async_smem();
    }
    tc::fence_before();
    __syncthreads();  // this item's shared tiles and tensor memory are free
    tc::fence_after();
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.R, 0, trow, sb + oTf);
        tc::tma_store_2d(&m.Rlo, 0, trow, sb + oT1);
        tc::bulk_commit();
    }
    }
    if (tid == STORE_TID) tc::bulk_wait_all();
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_prep_gdn(const Params& p, cudaStream_t s) {
    PrepGdnMaps m;
    const uint64_t T = (uint64_t)p.T_total;
    const uint64_t trows = (uint64_t)p.max_chunks * p.H * PD;  // rows of the [D][C] per chunk-head tiles
    const uint64_t crows = (uint64_t)p.max_chunks * p.H * CH;  // rows of the [C][C] per chunk-head tiles
    if (!(encode_tokens_map(&m.q, p.q, T, p.Hk, PD) && encode_tokens_map(&m.k, p.k, T, p.Hk, PD) &&
          encode_blocked_tokens_map(&m.v, p.v, T, p.H) && encode_rows_map(&m.W, p.W, trows, CH, PD) &&
          encode_rows_map(&m.U, p.U, trows, CH, PD) && encode_rows_map(&m.Kr, p.Kr, trows, CH, PD) &&
          encode_rows_map(&m.R, p.R, trows, CH, PD) && encode_rows_map(&m.Rlo, p.Rlo, trows, CH, PD) &&
          encode_rows_map(&m.T, p.Tm, crows, CH, CH)))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_prep_gdn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int items = p.max_chunks * p.H;
    const int ctas = items < num_sms() ? items : num_sms();
    k_prep_gdn<<<ctas, 512, SMEM_BYTES, s>>>(p, m);
    return cudaGetLastError();
}

}  // namespace gdr
