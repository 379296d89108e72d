// The two serial chunk recurrences on tcgen05 (D = 128), carried value-major:
// one CTA per (sequence, head, role) holds the whole transposed state S^T
// (128 value rows j x 128 key columns d) in fp32 registers of 8 consumer warps
// (thread = row j, 64 of the 128 columns) through every chunk of its sequence.
//
//   role 0, forward (chunk-start states, saved bf16 per chunk):
//       X^T = S0^T W^T ;  S_C^T = S0^T e^{gT} + (U - X)^T kr
//   role 1, backward (state gradient at each chunk end, saved bf16 per chunk; the
//       dh recurrence of "FlashQLA ... GDN 反向", §三, here transposed):
//       Y^T = dS_C^T kr^T ;  dS0^T = dS_C^T e^{gT} + dO^T (R_hi + R_lo) - Y^T W ;
//       dh0 = dS0 of the first chunk.
//
// Every product has M = 128 (the value rows), so every tensor-memory lane holds a
// useful row and the element-wise steps spread over all four SM sub-partitions.
// Per chunk: consumers write bf16 S^T into tensor memory, where it is the A operand of
// X^T (or Y^T) = S^T [C x D tile]^T; consumers write bf16 (U - X)^T (or -Y^T) into
// tensor memory, the A operand of the update product (role 1 also the state-independent
// dO^T R terms), which consumers add to the decayed state.  Both A operands stay in
// tensor memory (the thread of value row j owns lane j), so the chain's only shared
// operands are the chunk tiles.  A chain that saves its states also writes bf16 S^T to
// shared memory, off the chain's path, for a TMA store.  A separate TMA warp streams each
// chunk's tiles (and its e^{gT} row) two chunks ahead, refilling a stage when the
// products that read it have completed (one barrier per stage), and stores the saved
// states, so that neither issuing thread waits behind the other's instructions.  All
// waits are bounded; a wait that runs out sets a flag that turns every later wait and
// issue into a no-op, so all warps still meet every barrier and the CTA ends with its
// copies drained and its tensor memory released.
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"

namespace gdr {
namespace {

constexpr int SD = 128;
constexpr int TILE = CH * SD * 2;       // one C x D bf16 tile, 16 KB
constexpr int oEG = 5 * TILE;           // within a stage: e^{gT} row (fp32 [D])
constexpr int STAGE = 5 * TILE + 1024;  // role 0: W^T, kr^T, U^T ; role 1: kr^T, W^T, R_hi^T, R_lo^T, dO
// (the per-chunk tiles of the prep kernel are channel-major [D][C]; dO is token-major)
constexpr int oBS = 2 * STAGE;          // bf16 S^T [128 rows j][128 cols d]: the saved state's store source
constexpr int oBar = oBS + 2 * TILE;    // full[2], y, z, empty[2] mbarriers; tmem slot; abort flag
constexpr int SMEM_BYTES = oBar + 64 + 1024;
constexpr int NCONS = 256, NTHREADS = NCONS + 64;  // 8 consumer warps, the MMA warp, the TMA warp
constexpr int MMA_WARP = NCONS / 32, TMA_WARP = MMA_WARP + 1;
constexpr int N_PAIR = NCONS + 32;  // named barriers between the consumers and one of the other warps
// tensor-memory columns: Y^T / X^T (fp32), S^T (bf16 pairs, A operand), the update
// accumulators of the two stages (fp32), (U - X)^T / -Y^T (bf16 pairs, A operand)
constexpr uint32_t R_Y = 0, R_SA = 64, R_Z0 = 128, R_Z1 = 256, R_BA = 384;
// named barriers: S^T / the update operand ready (consumers -> MMA warp), the saved
// state's shared copy written (consumers -> TMA warp) and free again (TMA warp -> consumers)
constexpr int BAR_BS_READY = 1, BAR_BY_READY = 2, BAR_BS_FREE = 3, BAR_SAVE_READY = 4;

struct StateMaps {
    CUtensorMap W, Kr, Ut, R, Rlo, dO, S0, dS;
};

__device__ __forceinline__ int seq_chunk_begin(const Params& p, int seq) {
    if (p.chunk_off) return p.chunk_off[seq];
    return seq * (int)((p.seq_len + CH - 1) / CH);
}

// What one CTA runs: a chain over chunks [cb, ce) of one (sequence, head), walked upward
// (role 0) or downward (role 1), from a start state (zero, the identity, or a key-major
// [D][D] fp32 matrix), optionally saving the state entering each chunk, optionally with
// the chunks' input terms (U, or R^T dO) -- without them the chain multiplies the
// start state by the chunks' transitions -- and writing its final state key-major.
struct StateTask {
    int seq, h, role, cb, ce, input, save, identity;
    const float* init;
    float* out;
};

// Launch forms (phase, roles; roles: 1 = role 0, 2 = role 1, 3 = both):
//   phase 0  one chain per (sequence, head, asked role) over the whole sequence
//            (blockIdx.y picks the role when both are asked)
//   phase 1  segment phase 1, per (sequence, head): the role-0 chains of segments 0 .. G-2
//            (segment 0 from h0, the others from zero) and the role-1 chains of segments
//            1 .. G-1 (segment G-1 from dht, the others from zero), each if its role is
//            asked, and the transition chains of segments 1 .. G-2.  Segment 0 of role 0 and
//            segment G-1 of role 1 start from their true states here, so these two chains
//            save their per-chunk states in this phase.
//   phase 3  segment phase 3, per (sequence, head): the other segments of each asked role
//            (1 .. G-1 of role 0, 0 .. G-2 of role 1) from their true start states, saving
//            the per-chunk states (and dh0 / ht)
__host__ __device__ inline int phase1_tasks(int G, int roles) {
    return ((roles & 1) ? G - 1 : 0) + ((roles & 2) ? G - 1 : 0) + G - 2;
}
__device__ __forceinline__ StateTask decode_task(const Params& p, int phase, int roles) {
    StateTask t;
    const int G = p.seg_G, DD = 128 * 128;
    int pair, g = 0, kind = 0;  // kind: 0 data chain, 1 transition chain
    if (phase == 0) {
        pair = blockIdx.x;
        t.role = roles == 2 ? 1 : (int)blockIdx.y;
    } else if (phase == 1) {
        const int n0 = (roles & 1) ? G - 1 : 0, n1 = (roles & 2) ? G - 1 : 0;
        const int K = phase1_tasks(G, roles), k = blockIdx.x % K;
        pair = blockIdx.x / K;
        if (k < n0) {
            t.role = 0, g = k;
        } else if (k < n0 + n1) {
            t.role = 1, g = k - n0 + 1;
        } else {
            t.role = 0, g = k - n0 - n1 + 1, kind = 1;
        }
    } else {
        const int per = (roles == 3 ? 2 : 1) * (G - 1);
        pair = blockIdx.x / per;
        const int rem = blockIdx.x % per;
        t.role = roles == 3 ? rem / (G - 1) : (roles == 1 ? 0 : 1);
        g = rem % (G - 1) + (t.role == 0 ? 1 : 0);
    }
    t.seq = pair / p.H, t.h = pair % p.H;
    const int cb = seq_chunk_begin(p, t.seq), ce = seq_chunk_begin(p, t.seq + 1);
    const size_t pd = (size_t)pair * G;
    t.input = kind == 0;
    t.identity = kind == 1;
    // phase 1 saves along the two chains that start from their true states (h0, dht)
    t.save = phase != 1 || (kind == 0 && (t.role == 0 ? g == 0 : g == G - 1));
    t.out = nullptr;
    if (phase == 0) {
        t.cb = cb, t.ce = ce;
        t.init = t.role == 0 ? (p.h0 ? p.h0 + (size_t)pair * DD : nullptr) : (p.dht ? p.dht + (size_t)pair * DD : nullptr);
        if (t.role == 1) t.out = p.dh0 + (size_t)pair * DD;
        else if (p.ht) t.out = p.ht + (size_t)pair * DD;  // the forward's final state
    } else {
        const int len = (ce - cb + G - 1) / G;
        t.cb = min(cb + g * len, ce), t.ce = min(cb + (g + 1) * len, ce);
        const float* h0 = p.h0 ? p.h0 + (size_t)pair * DD : nullptr;
        const float* dht = p.dht ? p.dht + (size_t)pair * DD : nullptr;
        if (phase == 1) {
            t.init = kind == 1 ? nullptr : t.role == 0 ? (g == 0 ? h0 : nullptr) : (g == G - 1 ? dht : nullptr);
            t.out = (kind == 1 ? p.segP : t.role == 0 ? p.segL : p.segLb) + (pd + g) * DD;
        } else {
            if (t.role == 0)
                t.init = g == 0 ? h0 : p.segS + ((pd + g) * 2 + 0) * DD;
            else
                t.init = g == G - 1 ? dht : p.segS + ((pd + g) * 2 + 1) * DD;
            if (t.role == 1 && g == 0) t.out = p.dh0 + (size_t)pair * DD;
            if (t.role == 0 && g == G - 1 && p.ht) t.out = p.ht + (size_t)pair * DD;
        }
    }
    return t;
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1) k_states_tc(const Params p, int phase, int roles,
                                                           const __grid_constant__ StateMaps m) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);

    const StateTask task = decode_task(p, phase, roles);
    const int role = task.role, seq = task.seq, h = task.h;
    const int cb = task.cb, ce = task.ce;
    const int n = ce - cb;
    const int seq_cb = seq_chunk_begin(p, seq);  // the sequence's first chunk (token offsets)
    const int64_t bos = p.cu_seqlens ? p.cu_seqlens[seq] : (int64_t)seq * p.seq_len;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 6) + 1;
    const uint32_t full0 = smem_u32(bars), mby = smem_u32(bars + 2), mbz = smem_u32(bars + 3),
                   empty0 = smem_u32(bars + 4);

    if (warp == 0) tc::alloc(smem_u32(tslot), 512);
    if (tid == 0) {
        tc::mbar_init(full0, 1);
        tc::mbar_init(full0 + 8, 1);
        tc::mbar_init(mby, 1);
        tc::mbar_init(mbz, 1);
        tc::mbar_init(empty0, 1);
        tc::mbar_init(empty0 + 8, 1);
        *abort_flag = 0;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    auto failed = [&]() { return *abort_flag != 0; };
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!failed() && !tc::mbar_wait(bar, parity)) {
            *abort_flag = 1;
            atomicOr(p.status, ST_MMA_TIMEOUT);
        }
    };
    auto chunk_of = [&](int it) { return role == 0 ? cb + it : ce - 1 - it; };
    auto full_bar = [&](int it) { return full0 + 8 * (it & 1); };
    auto full_par = [&](int it) { return (uint32_t)((it >> 1) & 1); };

    if (warp == TMA_WARP) {
        // ---------------- TMA warp: tile loads two chunks ahead, saved-state stores ----------------
        int issued = 0;
        auto issue = [&](int it) {
            const int c = chunk_of(it);
            const uint32_t st = sb + (it & 1) * STAGE, bar = full_bar(it);
            const int row = (c * p.H + h) * CH;
            tc::mbar_expect_tx(bar, (task.input ? (role == 0 ? 3 : 5) : 2) * TILE + SD * 4);
            // channel-major tiles: 128 rows x 64 columns, one box each
            if (role == 0) {
                tc::tma_load_2d(st, &m.W, 0, 2 * row, bar);
                tc::tma_load_2d(st + TILE, &m.Kr, 0, 2 * row, bar);
                if (task.input) tc::tma_load_2d(st + 2 * TILE, &m.Ut, 0, 2 * row, bar);
            } else {
                tc::tma_load_2d(st, &m.Kr, 0, 2 * row, bar);
                tc::tma_load_2d(st + TILE, &m.W, 0, 2 * row, bar);
                tc::tma_load_2d(st + 2 * TILE, &m.R, 0, 2 * row, bar);
                tc::tma_load_2d(st + 3 * TILE, &m.Rlo, 0, 2 * row, bar);
                // rows past the sequence end are read too: they meet zero rows of R_hi / R_lo
                const int t0 = (int)(bos + (int64_t)(c - seq_cb) * CH);
                tc::tma_load_4d(st + 4 * TILE, &m.dO, 0, h, t0, 0, bar);
            }
            tc::bulk_load(st + oEG, p.egT + ((size_t)c * p.H + h) * SD, SD * 4, bar);
            issued = it + 1;
        };
        if (lane == 0) {
            tc::prefetch_map(&m.W);
            tc::prefetch_map(&m.Kr);
            tc::prefetch_map(role == 0 ? &m.Ut : &m.R);
            tc::prefetch_map(role == 0 ? &m.S0 : &m.Rlo);
            if (role == 1) {
                tc::prefetch_map(&m.dO);
                tc::prefetch_map(&m.dS);
            }
            if (n > 0) issue(0);
            if (n > 1) issue(1);
        }
        __syncwarp();
        if (task.save && n > 0) tc::named_arrive(BAR_BS_FREE, N_PAIR);
        for (int it = 0; it < n; ++it) {
            const int c = chunk_of(it);
            if (task.save) {  // store the state entering this step (S0 of chunk c, or dS_C of chunk c)
                tc::named_sync(BAR_SAVE_READY, N_PAIR);
                if (lane == 0) {
                    if (!failed()) {
                        tc::tma_store_3d(role == 0 ? &m.S0 : &m.dS, 0, (c * p.H + h) * SD, 0, sb + oBS);
                        tc::bulk_commit();
                    }
                    tc::bulk_wait_read();  // the shared copy may be rewritten
                }
                __syncwarp();
                if (it + 1 < n) tc::named_arrive(BAR_BS_FREE, N_PAIR);
            }
            if (lane == 0 && it + 2 < n) {
                // every product reading stage it & 1 has completed (its barrier completes once per
                // use of the stage, and the stage's next use needs the loads issued here, so the
                // wait cannot miss a phase)
                wait(empty0 + 8 * (it & 1), (uint32_t)((it >> 1) & 1));
                if (!failed()) issue(it + 2);
            }
            __syncwarp();
        }
        if (lane == 0) {
            // the last two loads issued are the newest phases of their barriers (drained on the failure path)
            for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i) tc::mbar_wait(full_bar(i), full_par(i));
            tc::bulk_wait_all();
        }
    } else if (warp == MMA_WARP) {
        // ---------------- MMA warp: every tcgen05.mma is issued by lane 0 ----------------
        // Role 1's state-independent products dO^T R_hi and dO^T R_lo fill the tensor pipe
        // while the consumers work: R_hi of a chunk right after its Y^T product (during the
        // element-wise step on Y), R_lo of the next chunk right after the update product
        // (during the state update); R_lo initialises the chunk's accumulator.
        constexpr uint32_t idr = tc::idesc(128, 128, 1, 0);
        auto r_part = [&](int j, int tile, uint32_t acc) {
            const uint32_t stj = sb + (j & 1) * STAGE, zj = tmem + ((j & 1) ? R_Z1 : R_Z0);
#pragma unroll
            for (int k = 0; k < CH; k += 16)
                tc::mma(zj, tc::mdesc(stj + 4 * TILE, CH, 0, k), tc::kdesc(stj + tile * TILE, SD, 0, k), idr,
                        acc || k > 0);
        };
        if (role == 1 && lane == 0 && n > 0) {
            wait(full_bar(0), full_par(0));
            if (!failed()) r_part(0, 3, 0);
        }
        for (int it = 0; it < n; ++it) {
            const uint32_t st = sb + (it & 1) * STAGE;
            const uint32_t z = tmem + ((it & 1) ? R_Z1 : R_Z0);
            tc::named_sync(BAR_BS_READY, N_PAIR);
            tc::fence_after();
            if (lane == 0) {
                wait(full_bar(it), full_par(it));
                if (!failed()) {
                    // X^T = S^T W^T (role 0) or Y^T = dS^T kr^T (role 1): A = S^T in tensor
                    // memory, B = the stage's first tile
                    constexpr uint32_t idy = tc::idesc(128, 64, 0, 1);
#pragma unroll
                    for (int k = 0; k < SD; k += 16)
                        tc::mma_ts(tmem + R_Y, tmem + R_SA + k / 2, tc::mdesc(st, SD, 0, k), idy, k > 0);
                    tc::commit(mby);
                    if (role == 1) r_part(it, 2, 1);  // + dO^T R_hi
                }
            }
            __syncwarp();
            tc::named_sync(BAR_BY_READY, N_PAIR);
            tc::fence_after();
            if (lane == 0 && !failed()) {
                // role 0: Z = (U - X)^T kr ; role 1: Z += (-Y^T) W   (A in tensor memory, B = the
                // stage's second tile)
                constexpr uint32_t idz = tc::idesc(128, 128, 0, 0);
#pragma unroll
                for (int k = 0; k < CH; k += 16)
                    tc::mma_ts(z, tmem + R_BA + k / 2, tc::kdesc(st + TILE, SD, 0, k), idz, role == 1 || k > 0);
                tc::commit(mbz);
                if (it + 2 < n) tc::commit(empty0 + 8 * (it & 1));  // the stage may be refilled
                if (role == 1 && it + 1 < n) {  // the next chunk's dO^T R_lo (its consumers read that buffer last step)
                    wait(full_bar(it + 1), full_par(it + 1));
                    if (!failed()) r_part(it + 1, 3, 0);
                }
            }
            __syncwarp();
        }
    } else {
        // ---------------- consumer warps: the state and the element-wise steps ----------------
        const int q4 = warp & 3, cg = warp >> 2;
        const int j = 32 * q4 + lane;  // tensor-memory lane = value row of S^T
        auto tl = [&](uint32_t col) { return tmem + ((uint32_t)(32 * q4) << 16) + col; };
        float S[64];  // S^T[j][64 cg + i], from the key-major start state (or zero, or the identity)
#pragma unroll
        for (int i = 0; i < 64; ++i)
            S[i] = task.init ? task.init[(size_t)(64 * cg + i) * SD + j] : (task.identity && 64 * cg + i == j ? 1.f : 0.f);
        for (int it = 0; it < n; ++it) {
            const unsigned char* stp = smem + (it & 1) * STAGE;
            const uint32_t z = (it & 1) ? R_Z1 : R_Z0;
            {
                // bf16 S^T[j][64 cg ..]: the A operand of this chunk's first product, in tensor memory
                uint32_t w0[16], w1[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    w0[e] = pack_bf16(S[2 * e], S[2 * e + 1]);
                    w1[e] = pack_bf16(S[32 + 2 * e], S[32 + 2 * e + 1]);
                }
                tc::st16u_nowait(tl(R_SA + 32 * cg), w0);
                tc::st16u_nowait(tl(R_SA + 32 * cg + 16), w1);
                tc::st_wait();
                tc::fence_before();
                tc::named_arrive(BAR_BS_READY, N_PAIR);
                if (task.save) {  // the same values to shared memory, the TMA store's source
                    tc::named_sync(BAR_BS_FREE, N_PAIR);
#pragma unroll
                    for (int jc = 0; jc < 4; ++jc) {
                        *reinterpret_cast<uint4*>(smem + oBS + tc::sw_chunk(j, 8 * cg + jc, SD)) =
                            make_uint4(w0[4 * jc], w0[4 * jc + 1], w0[4 * jc + 2], w0[4 * jc + 3]);
                        *reinterpret_cast<uint4*>(smem + oBS + tc::sw_chunk(j, 8 * cg + 4 + jc, SD)) =
                            make_uint4(w1[4 * jc], w1[4 * jc + 1], w1[4 * jc + 2], w1[4 * jc + 3]);
                    }
                    tc::fence_async_smem();
                    tc::named_arrive(BAR_SAVE_READY, N_PAIR);
                }
            }

            // this chunk's decay of the 64 columns (read before the stage can be refilled)
            wait(full_bar(it), full_par(it));
            float eg[64];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 v = *reinterpret_cast<const float4*>(stp + oEG + 4 * (64 * cg + 4 * i));
                eg[4 * i] = v.x;
                eg[4 * i + 1] = v.y;
                eg[4 * i + 2] = v.z;
                eg[4 * i + 3] = v.w;
            }
            wait(mby, it & 1);
            tc::fence_after();
            uint32_t wb[16];  // bf16 pairs of (U - X)^T or -Y^T, tokens 32 cg .. 32 cg + 31
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {  // tokens 32 cg + 16 qq .. +15
                float y[16];
                tc::ld16(tl(R_Y + 32 * cg + 16 * qq), y);
                const int jc = 4 * cg + 2 * qq;
                uint32_t w[8];
                if (role == 0 && task.input) {  // (U - X)^T
                    const uint4 u0 = *reinterpret_cast<const uint4*>(stp + 2 * TILE + tc::sw_chunk(j, jc, SD));
                    const uint4 u1 = *reinterpret_cast<const uint4*>(stp + 2 * TILE + tc::sw_chunk(j, jc + 1, SD));
                    const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 u = unpack_bf16(uw[e]);
                        w[e] = pack_bf16(u.x - y[2 * e], u.y - y[2 * e + 1]);
                    }
                } else {  // -Y^T (or -X^T of a transition chain)
#pragma unroll
                    for (int e = 0; e < 8; ++e) w[e] = pack_bf16(-y[2 * e], -y[2 * e + 1]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) wb[8 * qq + e] = w[e];
            }
            tc::st16u_nowait(tl(R_BA + 16 * cg), wb);
            tc::st_wait();
            tc::fence_before();
            tc::named_arrive(BAR_BY_READY, N_PAIR);

            wait(mbz, it & 1);
            tc::fence_after();
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                float zz[16];
                tc::ld16(tl(z + 64 * cg + 16 * qq), zz);
#pragma unroll
                for (int e = 0; e < 16; ++e) S[16 * qq + e] = fmaf(eg[16 * qq + e], S[16 * qq + e], zz[e]);
            }
            tc::fence_before();
        }
        if (task.out) {  // the final state, key-major [D][D] (dh0, or a segment's result)
#pragma unroll
            for (int i = 0; i < 64; ++i) task.out[(size_t)(64 * cg + i) * SD + j] = S[i];
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 512);
}

// Segment boundaries (phase 2), fp32 on CUDA cores: one CTA per (sequence, head, role,
// 16-column slice).  The columns of the state crossing a boundary are independent
// (S_end = P^T S_start + L acts on each column alone), so every slice walks the G - 1
// boundaries by itself; each output is summed over the key index in ascending order.
constexpr int CMB_COLS = 16, CMB_SLICES = 128 / CMB_COLS;
// 16-byte global -> shared copies that stay in flight together (LDGSTS), and the wait for them
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
__global__ void __launch_bounds__(256) k_seg_combine(const Params p, int roles) {
    extern __shared__ float sm[];
    float* tr = sm;               // [128][128] the segment's transition (P^T, key-major)
    float* cur = sm + 128 * 128;  // [128][16] this slice of the state crossing the boundary
    const int pair = blockIdx.x, role = roles == 3 ? (int)blockIdx.y : (roles == 1 ? 0 : 1), G = p.seg_G,
              DD = 128 * 128, j0 = CMB_COLS * (int)blockIdx.z;
    const size_t pd = (size_t)pair * G;
    // thread: rows 4 rb .. 4 rb + 3 and columns j0 + 2 cb, j0 + 2 cb + 1 of the slice; the
    // eight threads of a quarter warp share rb (their row reads are one broadcast)
    const int tid = threadIdx.x, rb = tid >> 3, cb = tid & 7;
    const float* first = role == 0 ? p.segL + (pd + 0) * DD : p.segLb + (pd + G - 1) * DD;
    for (int i = tid; i < 128 * CMB_COLS / 4; i += 256) {
        const int e = i / (CMB_COLS / 4), q = i % (CMB_COLS / 4);
        cp_async16(cur + 4 * i, first + e * 128 + j0 + 4 * q);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int step = 0; step < G - 1; ++step) {
        const int g = role == 0 ? step + 1 : G - 2 - step;  // the segment that starts from `cur`
        float* dst = p.segS + ((pd + g) * 2 + role) * DD;
        for (int i = tid; i < 128 * CMB_COLS / 4; i += 256) {
            const int e = i / (CMB_COLS / 4), q = i % (CMB_COLS / 4);
            *reinterpret_cast<float4*>(dst + e * 128 + j0 + 4 * q) = reinterpret_cast<const float4*>(cur)[i];
        }
        if (step == G - 2) break;  // the last segment's start is all phase 3 needs
        const float* P = p.segP + (pd + g) * DD;
        const float* L = (role == 0 ? p.segL : p.segLb) + (pd + g) * DD;
        // the whole transition in flight at once, this thread's part of L read meanwhile
#pragma unroll
        for (int u = 0; u < 128 * 128 / 4 / 256; ++u) cp_async16(tr + 4 * (tid + 256 * u), P + 4 * (tid + 256 * u));
        float acc[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float2 l2 = *reinterpret_cast<const float2*>(L + (size_t)(4 * rb + r) * 128 + j0 + 2 * cb);
            acc[r][0] = l2.x;
            acc[r][1] = l2.y;
        }
        cp_async_wait_all();
        __syncthreads();
#pragma unroll 2
        for (int e = 0; e < 128; e += 4) {
            float2 s[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] = *reinterpret_cast<const float2*>(cur + (e + u) * CMB_COLS + 2 * cb);
            if (role == 0) {  // (P^T S)[d][j] = sum_e P^T[d][e] S[e][j]
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float4 a = *reinterpret_cast<const float4*>(tr + (4 * rb + r) * 128 + e);
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc[r][0] = fmaf(av[u], s[u].x, acc[r][0]);
                        acc[r][1] = fmaf(av[u], s[u].y, acc[r][1]);
                    }
                }
            } else {          // (P dS)[d][j] = sum_e P^T[e][d] dS[e][j]
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 a = *reinterpret_cast<const float4*>(tr + (e + u) * 128 + 4 * rb);
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        acc[r][0] = fmaf(av[r], s[u].x, acc[r][0]);
                        acc[r][1] = fmaf(av[r], s[u].y, acc[r][1]);
                    }
                }
            }
        }
        __syncthreads();  // every read of cur and tr is done
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float2*>(cur + (4 * rb + r) * CMB_COLS + 2 * cb) = make_float2(acc[r][0], acc[r][1]);
        __syncthreads();
    }
}

// kernels that launch_states_tc launches for these directions (for the launch counts of
// gdr_profile_end): phase 1, the boundaries and phase 3 with segments, else one
int states_kernel_count(const Params& p, bool fwd, bool bwd) {
    if (!fwd && !bwd) return 0;
    return ((fwd && bwd) ? p.seg_G : p.seg_G1) >= 2 ? 3 : 1;
}

cudaError_t launch_states_tc(const Params& p, bool fwd, bool bwd, cudaStream_t s) {
    if (!fwd && !bwd) return cudaSuccess;
    StateMaps m;
    const uint64_t srows = (uint64_t)p.max_chunks * p.H * SD;  // D x D states
    bool ok = encode_rows_map(&m.W, p.W, srows, CH, SD) && encode_rows_map(&m.Kr, p.Kr, srows, CH, SD) &&
              encode_rows_map(&m.Ut, fwd ? p.U : nullptr, srows, CH, SD) &&
              encode_rows_map(&m.R, bwd ? p.R : nullptr, srows, CH, SD) &&
              encode_rows_map(&m.Rlo, bwd ? p.Rlo : nullptr, srows, CH, SD) &&
              encode_blocked_tokens_map(&m.dO, bwd ? p.dO : nullptr, (uint64_t)p.T_total, p.H) &&
              encode_blocked_rows_map(&m.S0, fwd ? p.S0 : nullptr, srows, SD) &&
              encode_blocked_rows_map(&m.dS, bwd ? p.dS : nullptr, srows, SD);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_states_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int pairs = p.N * p.H;
    const int roles = (fwd ? 1 : 0) | (bwd ? 2 : 0), nroles = roles == 3 ? 2 : 1;
    Params q = p;
    q.seg_G = roles == 3 ? p.seg_G : p.seg_G1;  // the segment count of this call's directions
    if (q.seg_G >= 2) {
        // time-parallel segments: phase 1 chains, the boundaries, phase 3 chains
        const int G = q.seg_G;
        k_states_tc<<<pairs * phase1_tasks(G, roles), NTHREADS, SMEM_BYTES, s>>>(q, 1, roles, m);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int cbytes = (128 * 128 + 128 * CMB_COLS) * 4;
        e = cudaFuncSetAttribute(k_seg_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, cbytes);
        if (e != cudaSuccess) return e;
        k_seg_combine<<<dim3(pairs, nroles, CMB_SLICES), 256, cbytes, s>>>(q, roles);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_states_tc<<<pairs * nroles * (G - 1), NTHREADS, SMEM_BYTES, s>>>(q, 3, roles, m);
        return cudaGetLastError();
    }
    k_states_tc<<<dim3(pairs, nroles), NTHREADS, SMEM_BYTES, s>>>(q, 0, roles, m);
    return cudaGetLastError();
}

}  // namespace gdr

