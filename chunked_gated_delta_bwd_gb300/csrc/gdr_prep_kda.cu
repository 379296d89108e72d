// Chunk-parallel preparation on tcgen05 for D = 128 with the per-channel (KDA) gate:
// persistent CTAs of 16 warps, one per SM, each looping over (chunk, head) items; the q, k,
// v tiles of the next item arrive by TMA into a second buffer while the current item is
// computed.  Its outputs are the per-chunk tiles of the state recurrences and the main
// backward (the X/R form of the FlashQLA dh kernel, "FlashQLA ... GDN 反向", §三; the
// scalar gate has its own kernel, gdr_prep_gdn.cu):
//
//   [A_raw; P] = [kd'; qd'] ki'^T       A = strict_lower(diag(beta) A_raw) (fp32), P = lower(.)
//                                        (a KDA backward also gets A (bf16) and P (a bf16
//                                        pair) for its main kernel, which needs both)
//   T   = (I + A)^-1                     (blocked inverse to fp32 accuracy, gdr_invert.cuh)
//   W^T = (beta kd)^T T^T                U^T = (beta V)^T T^T
//   R^T = qd^T - W^T P^T                 (a bf16 pair R_hi + R_lo)
//   kr  = kn e^{gT-gc}
//
// Products whose natural output is C x D are computed transposed (lane = channel), so
// a thread owns one channel for 16 rows; W, U, Kr, R_hi and R_lo are written
// channel-major ([D][C]), the layout the D = 128 state recurrence reads; T is written
// [C][C].  The raw q and k rows and e^{gc - ref} of the per-channel cumulative gate are
// staged in tensor memory once.
//
// The inverse runs on warps 0-7 while warps 8-15 build the T-independent operands of the
// next products.  The next item's beta logits and gate parameters are read one item ahead,
// its raw-gate tile by TMA into the space of the dead fp32 matrices.  W, U, Kr, R_hi and
// R_lo are staged in shared tiles that are dead by then and written by TMA stores, T from
// its bf16 shared tile (whose blocks above the diagonal stay zero).
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"
#include "gdr_invert.cuh"

namespace gdr {

namespace {

constexpr int PD = 128;
constexpr int TILE = CH * PD * 2;  // 16 KB
using inv::LDF;
using inv::XLD;
// shared-memory map (bytes from the 1024-aligned base); two input stages of q, k, v
constexpr int STAGE = 3 * TILE;
constexpr int oQ = 0;         // q (token-major) -> (beta kd)^T [d][s]   (+ STAGE for the other stage)
constexpr int oK = 16384;     // k (token-major) -> (beta V)^T [j][s]
constexpr int oV = 32768;     // v (token-major)
constexpr int oW0 = 2 * STAGE;  // kd'^T [d][r] (G1, A block 0) -> (KDA backward) A, P lo [r][s] bf16 staged
                                //   -> R_lo^T staged
constexpr int oW1 = oW0 + TILE; // qd'^T [d][r] (G1, A block 1) -> R_hi^T staged
constexpr int oW2 = oW1 + TILE; // ki'^T [d][s] (G1, B) -> W^T bf16 [d][s]
constexpr int oP = oW2 + TILE;  // P [r][s] bf16
constexpr int oT = oP + 8192;   // T [r][s] bf16
constexpr int oA = oT + 8192;   // A fp32 [64][LDF] row-major; the next item's raw gates before
constexpr int oTf = oA + CH * LDF * 4;  // T fp32, transposed [c][r], stride LDF
constexpr int oTmp = oTf + CH * LDF * 4;  // 8 warps' transfer tiles [8][XLD]
constexpr int nTmp = 8 * 8 * XLD;
constexpr int oGR = (oTmp + nTmp * 4 + 1023) / 1024 * 1024;  // raw gates (token-major) of the item
static_assert(oTmp + nTmp * 4 <= oGR, "inversion scratch overlaps the raw-gate tile");
constexpr int oSmall = oGR + TILE;
static_assert(nTmp >= 4 * PD, "the gate scan's minima fit the transfer tiles");
constexpr int nInvQ = 64, nInvK = 64, nBeta = 64, nFac = 256, nRef = 128, nGT = 128, nScan = 512;
constexpr int SMALL_FLOATS = nInvQ + nInvK + nBeta + nFac + nRef + nGT + nScan;
constexpr int SMEM_BYTES = oSmall + SMALL_FLOATS * 4 + 128 + 1024;  // + barriers, tensor-memory slot, chunk info
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
constexpr uint32_t R_G1 = 0, R_W = 64, R_U = 128, R_R = 192, R_Q = 256, R_K = 320, R_G = 384;

struct PrepMaps {
    CUtensorMap q, k, v, graw, W, U, Kr, R, Rlo, T, ap;
};
// The thread that issues the TMA stores of W, U, Kr, R_hi, R_lo and T and the copies of the
// next item's q, k and v: its stores read the stage that those copies overwrite, and a
// bulk store's completion is visible only to the thread that issued it.
constexpr int STORE_TID = 416;

}  // namespace

template <int GATE>
__global__ void __launch_bounds__(512, 1) k_prep_kda(const Params p, const __grid_constant__ PrepMaps m) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // items (chunk, head) = chunk * H + h over the chunks that exist
    const int total_chunks = p.chunk_off ? p.chunk_off[p.N] : p.N * (int)((p.seq_len + CH - 1) / CH);
    const int n_items = total_chunks * p.H;
    const int q4 = warp & 3, hc = warp >> 2;
    const int L = 32 * q4 + lane;  // this thread's lane: a channel, or a stacked row of G1
    const int c0 = 16 * hc;        // first of this thread's 16 rows

    unsigned char *sW0 = smem + oW0, *sW1 = smem + oW1, *sW2 = smem + oW2, *sP = smem + oP, *sT = smem + oT;
    float* sA = reinterpret_cast<float*>(smem + oA);
    float* sTf = reinterpret_cast<float*>(smem + oTf);
    float* sTmp = reinterpret_cast<float*>(smem + oTmp);
    float* fsm = reinterpret_cast<float*>(smem + oSmall);
    float* sInvQ = fsm;
    float* sInvK = sInvQ + nInvQ;
    float* sBeta = sInvK + nInvK;
    float* sFac = sBeta + nBeta;  // [2][128] e^{ref}, e^{gT-ref} per channel
    float* sRef = sFac + nFac;    // ref[d]
    float* sGT = sRef + nRef;     // gT[d]
    float* sScan = sGT + nGT;     // [4][128]
    uint64_t* mbars = reinterpret_cast<uint64_t*>(sScan + nScan);
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
    const uint32_t mb = smem_u32(mbars), mload0 = smem_u32(mbars + 1);  // load barriers: one per stage
    const uint32_t mgr = smem_u32(mbars + 3);                            // the raw-gate tile

    // q, k, v of item `it` into stage s: copy `which` (0 q, 1 k, 2 v) or all (which < 0); the
    // copies may be issued by different threads in any order (the barrier's transaction
    // count can run ahead of the expectation registered with copy 0)
    auto issue_loads = [&](int item, const ChunkInfo& cj, int stg, int which) {
        const int hh = item % p.H, t0 = (int)cj.t0;
        const uint32_t bar = mload0 + 8 * stg, st = sb + stg * STAGE;
        if (which <= 0) {
            tc::mbar_expect_tx(bar, 3 * TILE);
            tc::tma_load_4d(st + oQ, &m.q, 0, qk_head(p, hh), t0, 0, bar);
        }
        if (which < 0 || which == 1) tc::tma_load_4d(st + oK, &m.k, 0, qk_head(p, hh), t0, 0, bar);
        if (which < 0 || which == 2) tc::tma_load_4d(st + oV, &m.v, 0, hh, t0, 0, bar);
    };
    // raw gates of `item`, token-major, into their own tile (requested as soon as the item
    // before has read its gates, a whole item ahead of their use)
    auto issue_gate_load = [&](int item, const ChunkInfo& cj) {
        tc::mbar_expect_tx(mgr, TILE);
        tc::tma_load_4d(sb + oGR, &m.graw, 0, item % p.H, (int)cj.t0, 0, mgr);
    };
    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) {
        tc::mbar_init(mb, 1);
        tc::mbar_init(mload0, 1);
        tc::mbar_init(mload0 + 8, 1);
        tc::mbar_init(mgr, 1);
        for (int j = 0; j < 2; ++j) {  // the first two items' chunk info
            ChunkInfo c{};
            if ((int)blockIdx.x + j * (int)gridDim.x < n_items)
                lookup_chunk(((int)blockIdx.x + j * (int)gridDim.x) / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, c);
            put_ci(j, c);
            if (j == 0 && (int)blockIdx.x < n_items) {
                issue_loads(blockIdx.x, c, 0, -1);
                issue_gate_load(blockIdx.x, c);
            }
        }
    }
    // T's blocks above the diagonal stay zero in the shared tile
    for (int i = tid; i < CH * CH * 2 / 16; i += 512)
        *reinterpret_cast<uint4*>(smem + oT + 16 * i) = make_uint4(0, 0, 0, 0);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    uint32_t phase = 0;
    int it = 0;  // this CTA's item count (selects the stage)
    auto tl = [&](uint32_t col) { return tmem + ((uint32_t)(32 * q4) << 16) + col; };
    auto sync_all = [&]() {
        tc::fence_async_smem();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    int pending = -1;  // stage with a load in flight that this item does not consume, or -1
    uint32_t pending_par = 0;
    bool pending_g = (int)blockIdx.x < n_items;  // a raw-gate tile is in flight ...
    uint32_t pend_g_par = 0;                       // ... completing this phase parity of its barrier
    auto bail = [&]() {
        if (tid == 0) {
            atomicOr(p.status, ST_MMA_TIMEOUT);
            if (pending >= 0) tc::mbar_wait(mload0 + 8 * pending, pending_par);  // bounded drain
            if (pending_g) tc::mbar_wait(mgr, pend_g_par);
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
    // the next item's beta logit (thread r < 64) and gate parameters (every thread: its
    // channel), read one item ahead as raw values (row clamped into the chunk) that are
    // first read at the next item's top, so no thread waits for them
    float pbias = 0.f, palog = 0.f;
    unsigned short pb = 0;
    auto prefetch_small = [&](int item, const ChunkInfo& cj) {
        const int hh = item % p.H;
        if (tid < CH)
            pb = reinterpret_cast<const unsigned short*>(p.beta_logit)[(cj.t0 + min(tid, cj.len - 1)) * p.H + hh];
        pbias = p.dt_bias[hh * PD + L];
        palog = p.A_log[hh];
    
    };
    if ((int)blockIdx.x < n_items) prefetch_small(blockIdx.x, get_ci(0));  // (slot written before the barrier above)
    // a[cq .. cq+15]
    auto rows16 = [&](const float* a, float (&o)[16], int cq) {
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

    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const int chunk = item / p.H, h = item % p.H;
    const int stg = it & 1;
    const ChunkInfo ci = get_ci(stg);
    unsigned char *sQ = smem + stg * STAGE + oQ, *sK = smem + stg * STAGE + oK, *sV = smem + stg * STAGE + oV;
    const uint32_t sQa = sb + stg * STAGE + oQ, sKa = sb + stg * STAGE + oK;
    const size_t tile_cc = ((size_t)chunk * p.H + h) * CH * CH;
    const bool has_next = item + (int)gridDim.x < n_items;
    pending = -1;  // (the next item's tiles are requested while this item is inverted)
    if (tid < CH) sBeta[tid] = tid < ci.len ? sigmoid_f(__bfloat162float(__ushort_as_bfloat16(pb))) : 0.f;

    // per-channel log gates of this thread's channel and rows (raw gates from the
    // token-major tile in the space of A), scanned across the four row quarters, staged in
    // tensor memory; the gate-range check of the chunk
    float refL = 0.f, gTL = 0.f;
    {
        const float a = expf(palog);
        const float bias = pbias;
        if (has_next) prefetch_small(item + gridDim.x, get_ci(stg ^ 1));  // raw values, first read at the next item's top
        {
            const bool ok = tc::mbar_wait(mgr, (uint32_t)(it & 1));
            if (__syncthreads_or(!ok)) return bail();
            pending_g = false;
        }
        float g[16];
        {
            const unsigned char* gt = smem + oGR;
            const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
                g[i] = c0 + i < ci.len ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(gt + off)) : 0.f;
            }
        }
        // the quarter's scan, its total and extrema; one exchange gives every thread the
        // prefix, the chunk total and the chunk's extrema of its channel (the maximum over
        // the rows is the largest quarter maximum plus that quarter's prefix, bit for bit:
        // fp32 addition is monotone)
        float acc = 0.f, lmx = -3.0e38f, lmn = 3.0e38f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (c0 + i < ci.len) acc += kda_gate_fn<GATE>(p.gate_scale, a, g[i] + bias);
            g[i] = acc;
            lmx = fmaxf(lmx, acc);
            lmn = fminf(lmn, acc);
        }
        sScan[hc * PD + L] = acc;
        sTmp[hc * PD + L] = lmx;  // the inversion scratch is not in use yet
        sTmp[4 * PD + hc * PD + L] = lmn;
        __syncthreads();
        if (has_next) {  // every thread has read this item's raw gates: the next item's, into the tile
            if (tid == 480) issue_gate_load(item + gridDim.x, get_ci(stg ^ 1));  // (not the product-issuing thread)
            pending_g = true;
            pend_g_par = (uint32_t)((it + 1) & 1);
        }
        float pre = 0.f, tot = 0.f, M = -3.0e38f, N = 3.0e38f;
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
            const float t = sScan[h2 * PD + L];
            M = fmaxf(M, tot + sTmp[h2 * PD + L]);
            N = fminf(N, tot + sTmp[4 * PD + h2 * PD + L]);
            if (h2 < hc) pre += t;
            tot += t;
        }
        refL = 0.5f * (M + N);
        gTL = tot;
        // e^{gc - ref} of this thread's channel and rows, in tensor memory
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = __expf((g[i] + pre) - refL);
        tc::st16(tl(R_G + c0), g);
        if (hc == 0) {
            sRef[L] = refL;
            sGT[L] = tot;
            sFac[L] = __expf(refL);             // e^{ref}
            sFac[PD + L] = __expf(tot - refL);  // e^{gT - ref}
            if (0.5f * (M - N) > 80.f || M > 80.f) atomicOr(p.status, ST_GATE_RANGE);
        }
    }

    // operand tiles; rows past the chunk's end read as zero
    {
        const bool ok = tc::mbar_wait(mload0 + 8 * stg, (uint32_t)((it >> 1) & 1));
        if (__syncthreads_or(!ok)) return bail();
    }
    if (ci.len < CH) {
        const int nz = (CH - ci.len) * 16;
        for (int i = tid; i < 3 * nz; i += 512) {
            const int t = i / nz, rem = i % nz, r = ci.len + rem / 16, jc = rem % 16;
            unsigned char* base = t == 0 ? sQ : t == 1 ? sK : sV;
            *reinterpret_cast<uint4*>(base + tc::sw_chunk(r, jc, 64)) = make_uint4(0, 0, 0, 0);
        }
    }
    __syncthreads();
    {  // inverse row norms of q and k, 4 threads per row
        const int r = (tid >> 2) & 63, part = tid & 3;
        const unsigned char* src = tid < 256 ? sQ : sK;
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
    {  // raw q and k of this thread's channel and rows into tensor memory
        const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
        float qs[16], ks[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (c0 + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
            qs[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sQ + off));
            ks[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sK + off));
        }
        tc::st16(tl(R_Q + c0), qs);
        tc::st16(tl(R_K + c0), ks);
    }
    // the last item's stores have read their shared tiles: the R store (the G1 operand tiles,
    // rewritten below) and the T store (sT, which this item's inversion rewrites).  Both
    // orderings rest on this one full wait: a narrower form (one store still reading) would
    // let the next inversion overwrite T while its store is in flight.
    if (tid == STORE_TID) tc::bulk_wait_read();
    __syncthreads();  // norms, factors and the q / k tile reads are done

    // gate factors of this thread's channel and rows cq .. cq+15
    auto factors = [&](int kind, float (&f)[16], int cq) {
        {
            // e^{gc-ref} from tensor memory; e^{gc} = e^{gc-ref} e^{ref}, e^{ref-gc} = 1 / e^{gc-ref},
            // e^{gT-gc} = e^{gT-ref} / e^{gc-ref} (|gc - ref| <= 80: no overflow)
            const float eRef = sFac[L], eGTref = sFac[PD + L];
            float e[16];
            tc::ld16(tl(R_G + cq), e);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (kind == F_KDP) f[i] = e[i];
                else if (kind == F_KD) f[i] = e[i] * eRef;
                else if (kind == F_KIP) f[i] = __fdividef(1.f, e[i]);
                else f[i] = __fdividef(eGTref, e[i]);
            }
        }
    };
    // x (raw q or k of this channel and rows cq ..) * m_r * f, m_r = inv_r * mul * rowmul_r
    auto derived = [&](bool isq, float mul, const float* rowmul, int kind, float (&o)[16], int cq) {
        float f[16], inv[16], rm[16];
        factors(kind, f, cq);
        tc::ld16(tl((isq ? R_Q : R_K) + cq), o);
        rows16(isq ? sInvQ : sInvK, inv, cq);
        if (rowmul) rows16(rowmul, rm, cq);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = o[i] * derived_m(inv[i], mul, rowmul ? rm[i] : 1.f) * f[i];
    };
    auto build = [&](unsigned char* tile, bool isq, float mul, const float* rowmul, int kind, int cq) {
        float v[16];
        uint32_t w[8];
        derived(isq, mul, rowmul, kind, v, cq);
        pack8(v, w);
        store_cm(tile, w, cq);
    };

    // ---- G1: [A_raw; P] = [kd'; qd'] ki'^T ----------------------------------------------
    build(sW0, false, 1.f, nullptr, F_KDP, c0);
    build(sW1, true, p.scale, nullptr, F_KDP, c0);
    build(sW2, false, 1.f, nullptr, F_KIP, c0);
    sync_all();
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 1, 1);
#pragma unroll
        for (int k = 0; k < PD; k += 16)
            tc::mma(tmem + R_G1, tc::mdesc(sb + oW0, 128, 0, k), tc::mdesc(sb + oW2, 128, 0, k), id, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    {
        float v[16];
        tc::ld16(tl(R_G1 + c0), v);
        // (the KDA backward also takes A and P for its main kernel, which then needs no first
        // product of its own: A and P lo are staged [r][s] bf16 in the dead kd' tile, P hi is
        // sP, and one thread stores the three below)
        const bool ap = p.APm != nullptr;
        if (L < 64) {  // A = strict_lower(beta A_raw), fp32 for the inversion
            const int r = L;
            const float br = sBeta[r];
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = c0 + i < r ? br * v[i] : 0.f;
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(sA + r * LDF + c0 + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
            if (ap) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = pack_bf16(a[2 * e], a[2 * e + 1]);
                *reinterpret_cast<uint4*>(sW0 + tc::sw_chunk(r, c0 >> 3, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(sW0 + tc::sw_chunk(r, (c0 >> 3) + 1, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        } else {  // P = lower(qd' ki'^T), bf16 [r][s]
            const int r = L - 64;
            uint32_t w[8];
            float pv[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s0 = c0 + 2 * e;
                pv[2 * e] = s0 <= r ? v[2 * e] : 0.f;
                pv[2 * e + 1] = s0 + 1 <= r ? v[2 * e + 1] : 0.f;
                w[e] = pack_bf16(pv[2 * e], pv[2 * e + 1]);
            }
            *reinterpret_cast<uint4*>(sP + tc::sw_chunk(r, c0 >> 3, 64)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(sP + tc::sw_chunk(r, (c0 >> 3) + 1, 64)) = make_uint4(w[4], w[5], w[6], w[7]);
            if (p.Pm) {  // forward output: P [r][s] per chunk-head
                uint4* g = reinterpret_cast<uint4*>(p.Pm + tile_cc + r * CH + c0);
                g[0] = make_uint4(w[0], w[1], w[2], w[3]);
                g[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            if (ap) {  // P's residual P - hi (P hi is sP)
                uint32_t wl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 hf = unpack_bf16(w[e]);
                    wl[e] = pack_bf16(pv[2 * e] - hf.x, pv[2 * e + 1] - hf.y);
                }
                unsigned char* lo = sW0 + CH * CH * 2;
                *reinterpret_cast<uint4*>(lo + tc::sw_chunk(r, c0 >> 3, 64)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                *reinterpret_cast<uint4*>(lo + tc::sw_chunk(r, (c0 >> 3) + 1, 64)) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
            }
        }
        if (ap) tc::fence_async_smem();  // the staged tiles (and sP) go out by TMA after the barrier
    }
    __syncthreads();
    if (p.APm && tid == STORE_TID) {  // A, P hi, P lo for the main kernel, one group of stores
        const int row = 3 * (chunk * p.H + h) * CH;
        tc::tma_store_2d(&m.ap, 0, row, sb + oW0);
        tc::tma_store_2d(&m.ap, 0, row + CH, sb + oP);
        tc::tma_store_2d(&m.ap, 0, row + 2 * CH, sb + oW0 + CH * CH * 2);
        tc::bulk_commit();
    }
    if (warp < 8) {
        inv::invert_tc(sA, sTf, sTmp, sT, nullptr);
        // (warps 6, 7 leave the inversion after its diagonal blocks) the chunk info of the item
        // after next, into this item's slot
        if (tid == 192 && item + 2 * (int)gridDim.x < n_items) {
            ChunkInfo c2;
            lookup_chunk((item + 2 * (int)gridDim.x) / p.H, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, c2);
            put_ci(stg, c2);
        }
    } else {
        // (beta kd)^T -> the q tile's space ; (beta V)^T -> the k tile's space; this warp's
        // lanes for row quarters (hc - 2) and hc
        for (int pass = 0; pass < 2; ++pass) {
            const int cq = 16 * (hc - 2 + 2 * pass);
            build(sQ, false, 1.f, sBeta, F_KD, cq);
            float v[16], bt[16];
            uint32_t w[8];
            rows16(sBeta, bt, cq);
            const int lch = (L & 63) >> 3, lsub = (L & 7) << 1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t off = (uint32_t)((L >> 6) * 64 * 128 + (cq + i) * 128 + ((lch ^ (i & 7)) << 4) + lsub);
                v[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sV + off)) * bt[i];
            }
            pack8(v, w);
            store_cm(sK, w, cq);
        }
        // the next item's tiles into the other stage, once the last item's stores have read it
        // (its R_hi, R_lo store, the latest group, reads no stage)
        if (has_next) {
            if (tid == STORE_TID) {
                tc::bulk_wait_read_but1();
                issue_loads(item + gridDim.x, get_ci(stg ^ 1), stg ^ 1, -1);
            }
            pending = stg ^ 1;
            pending_par = (uint32_t)(((it + 1) >> 1) & 1);
        }
    }
    sync_all();
    if (tid == STORE_TID) {  // T for the main backward (its blocks above the diagonal stay zero in the tile);
                             // the next item's inversion rewrites sT only after the full read wait
                             // of the store thread at that item's top
        tc::tma_store_2d(&m.T, 0, (chunk * p.H + h) * CH, sb + oT);
        tc::bulk_commit();
    }

    // ---- W^T = (beta kd)^T T^T ; U^T = (beta V)^T T^T --------------------------------------
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 0, 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_W, tc::kdesc(sQa, 128, 0, k), tc::kdesc(sb + oT, 64, 0, k), id, k > 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_U, tc::kdesc(sKa, 128, 0, k), tc::kdesc(sb + oT, 64, 0, k), id, k > 0);
        tc::commit(mb);
    }
    if (!wait_mma()) return;
    const int trow = (chunk * p.H + h) * PD;  // the chunk-head's first row in the [D][C] tile maps
    {
        float v[16];
        uint32_t w[8];
        tc::ld16(tl(R_W + c0), v);
        pack8(v, w);
        store_cm(sW2, w, c0);  // bf16 W^T, the A operand of W^T P^T (ki' is dead) and W's store
        tc::ld16(tl(R_U + c0), v);
        pack8(v, w);
        store_cm(sK, w, c0);  // U^T over the dead (beta V)^T
    }
    sync_all();
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.W, 0, trow, sb + oW2);
        tc::tma_store_2d(&m.U, 0, trow, sKa);
        tc::bulk_commit();
        // (KDA backward) the A / P stores, two groups back, have read the kd' tile, where R_lo
        // is staged next, and sP; the wait of the next product orders this for every thread
        if (p.APm) tc::bulk_wait_read_but1();
    }

    // ---- R^T = qd^T - W^T P^T ----------------------------------------------------------------
    if (tid == 0) {
        constexpr uint32_t id = tc::idesc(128, 64, 0, 0);
#pragma unroll
        for (int k = 0; k < CH; k += 16)
            tc::mma(tmem + R_R, tc::kdesc(sb + oW2, 128, 0, k), tc::kdesc(sb + oP, 64, 0, k), id, k > 0);
        tc::commit(mb);
    }
    // while the tensor cores run: kr = kn e^{gT-gc} (over the dead v tile) ; gT, e^{gT}
    {
        float v[16];
        uint32_t w[8];
        derived(false, 1.f, nullptr, F_KR, v, c0);
        pack8(v, w);
        store_cm(sV, w, c0);
        tc::fence_async_smem();
        if (hc == 0) {
            const float gt = gTL;
            p.gT[((size_t)chunk * p.H + h) * PD + L] = gt;
            p.egT[((size_t)chunk * p.H + h) * PD + L] = __expf(gt);
        }
    }
    if (!wait_mma()) return;
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.Kr, 0, trow, sb + stg * STAGE + oV);
        tc::bulk_commit();
    }
    {
        float acc[16], qd[16];
        uint32_t w[8], wl[8];
        tc::ld16(tl(R_R + c0), acc);
        derived(true, p.scale, nullptr, F_KD, qd, c0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float r0 = qd[2 * e] - acc[2 * e], r1 = qd[2 * e + 1] - acc[2 * e + 1];
            w[e] = pack_bf16(r0, r1);
            const float2 hf = unpack_bf16(w[e]);
            wl[e] = pack_bf16(r0 - hf.x, r1 - hf.y);
        }
        store_cm(sW1, w, c0);  // R_hi over the dead qd'^T
        store_cm(sW0, wl, c0);  // R_lo over the dead kd'^T
        tc::fence_async_smem();
    }
    tc::fence_before();
    __syncthreads();  // this item's shared tiles and tensor memory are free
    tc::fence_after();
    if (tid == STORE_TID) {
        tc::tma_store_2d(&m.R, 0, trow, sb + oW1);
        tc::tma_store_2d(&m.Rlo, 0, trow, sb + oW0);
        tc::bulk_commit();
    }
    }
    if (tid == STORE_TID) tc::bulk_wait_all();
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

template <int GATE>
static cudaError_t launch_prep_kda_t(const Params& p, cudaStream_t s) {
    PrepMaps m;
    const uint64_t T = (uint64_t)p.T_total;
    const uint64_t trows = (uint64_t)p.max_chunks * p.H * PD;  // rows of the [D][C] per chunk-head tiles
    const uint64_t crows = (uint64_t)p.max_chunks * p.H * CH;  // rows of the [C][C] per chunk-head tiles
    if (!(encode_blocked_tokens_map(&m.q, p.q, T, p.Hk) && encode_blocked_tokens_map(&m.k, p.k, T, p.Hk) &&
          encode_blocked_tokens_map(&m.v, p.v, T, p.H) &&
          encode_blocked_tokens_map(&m.graw, p.g_raw, T, p.H) &&
          encode_rows_map(&m.W, p.W, trows, CH, PD) && encode_rows_map(&m.U, p.U, trows, CH, PD) &&
          encode_rows_map(&m.Kr, p.Kr, trows, CH, PD) && encode_rows_map(&m.R, p.R, trows, CH, PD) &&
          encode_rows_map(&m.Rlo, p.Rlo, trows, CH, PD) && encode_rows_map(&m.T, p.Tm, crows, CH, CH) &&
          encode_rows_map(&m.ap, p.APm, 3 * crows, CH, CH)))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_prep_kda<GATE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int items = p.max_chunks * p.H;
    const int ctas = items < num_sms() ? items : num_sms();
    k_prep_kda<GATE><<<ctas, 512, SMEM_BYTES, s>>>(p, m);
    return cudaGetLastError();
}

cudaError_t launch_prep_kda(const Params& p, cudaStream_t s) {
    // the KDA gate function is a template parameter: each instance carries only its own code
    return p.kda_gate == 0 ? launch_prep_kda_t<0>(p, s) : launch_prep_kda_t<1>(p, s);
}

}  // namespace gdr
