// The two serial chunk recurrences, one CTA per (sequence, head, value slice).
//
// The state S (dk x dv) and its gradient dS are independent across value
// columns, so each CTA (8 warps) owns BV = 32 columns and carries them in
// fp32 registers through every chunk of its sequence.  Both recurrences use only
// the per-chunk tiles written by the prep kernel; neither depends on the
// other, so one launch runs both (blockIdx.y selects the role).
//
//   role 0, forward  (chunk-start states, saved bf16 per chunk, value-major):
//       X = W S0 ;  S_C = diag(e^{gT}) S0 + kr^T (U - X)
//   role 1, backward (state gradient at each chunk end, saved bf16 per chunk;
//       the FlashQLA dh recurrence, "FlashQLA ... GDN 反向", §三):
//       Y = kr dS_C ;  dS0 = diag(e^{gT}) dS_C + (R_hi + R_lo)^T dO - W^T Y
//       and dh0 = dS0 of each sequence's first chunk (fp32).
#include "gdr_chunk.cuh"

namespace gdr {

constexpr int BV = 32;        // value columns per CTA
constexpr int LDV = BV + 8;   // padded row (elements) of the narrow tiles

template <int D>
struct StateSmem {
    static constexpr int ROWB = 2 * D;
    static constexpr int TCD = CH * ROWB;
    static constexpr int TNV = CH * LDV * 2;  // C x BV narrow tile
    // one stage: four C x D tiles, one narrow tile, gT
    static constexpr int oT0 = 0, oT1 = TCD, oT2 = 2 * TCD, oT3 = 3 * TCD, oN = 4 * TCD, oG = oN + TNV,
                         stage = oG + D * 4;
    static constexpr int oStage0 = 0, oStage1 = stage, oS = 2 * stage, oY = oS + D * LDV * 2,
                         bytes = oY + TNV;
};

template <int D>
__device__ __forceinline__ int chunk_begin(const Params& p, int seq) {
    if (p.chunk_off) return p.chunk_off[seq];
    return seq * (int)((p.seq_len + CH - 1) / CH);
}

template <int D>
__global__ void __launch_bounds__(256) k_states(const Params p, int role0) {
    using SM = StateSmem<D>;
    using TileCD = SwzTile<SM::ROWB>;
    using TileN = PadTile<LDV>;
    constexpr int SLICES = D / BV;
    constexpr int MT = D / 64;  // 16-row tiles per warp over the dk rows (4 row bands x 2 column halves)
    extern __shared__ __align__(1024) unsigned char smem[];

    const int role = role0 + blockIdx.y;
    const int slice = blockIdx.x % SLICES;
    const int pair = blockIdx.x / SLICES;
    const int seq = pair / p.H, h = pair % p.H;
    const int cb = chunk_begin<D>(p, seq), ce = chunk_begin<D>(p, seq + 1);
    const int warp = threadIdx.x >> 5;
    const int col0 = slice * BV;
    const int64_t bos = p.cu_seqlens ? p.cu_seqlens[seq] : (int64_t)seq * p.seq_len;
    const int64_t eos = p.cu_seqlens ? p.cu_seqlens[seq + 1] : bos + p.seq_len;

    TileN sS{smem + SM::oS}, sY{smem + SM::oY};
    auto stage = [&](int b) { return smem + (b ? SM::oStage1 : SM::oStage0); };

    // state fragment of this warp: rows 16*MT*(warp&3) .. (D/4 rows), columns 16*(warp>>2) .. +16
    const int m0 = 16 * MT * (warp & 3), n0 = 16 * (warp >> 2);
    const int mx = 16 * (warp & 3);  // rows of the C x BV product
    float st[MT][2][4];
    {
        const float* init = role == 0 ? p.h0 : p.dht;
        const size_t sb = ((size_t)seq * p.H + h) * D * D;
        frag_foreach(st, m0, n0, [&](int r, int c, float& a0, float& a1) {
            a0 = init ? init[sb + (size_t)r * D + col0 + c] : 0.f;
            a1 = init ? init[sb + (size_t)r * D + col0 + c + 1] : 0.f;
        });
    }

    // loads of one chunk's operands into a stage
    auto issue = [&](int c, int b) {
        unsigned char* s = stage(b);
        const size_t tcd = ((size_t)c * p.H + h) * CH * D;
        TileCD t0{s + SM::oT0}, t1{s + SM::oT1}, t2{s + SM::oT2}, t3{s + SM::oT3};
        TileN tn{s + SM::oN};
        if (role == 0) {
            async_load_tile<CH, D>(t0, p.W + tcd);
            async_load_tile<CH, D>(t1, p.Kr + tcd);
            for (int i = threadIdx.x; i < CH * (BV / 8); i += blockDim.x) {
                const int r = i / (BV / 8), j = i % (BV / 8);
                cp_async16(tn.chunk(r, j), p.U + tcd + r * D + col0 + j * 8, true);
            }
        } else {
            async_load_tile<CH, D>(t0, p.Kr + tcd);
            async_load_tile<CH, D>(t1, p.R + tcd);
            async_load_tile<CH, D>(t2, p.W + tcd);
            async_load_tile<CH, D>(t3, p.Rlo + tcd);
            const int local = c - cb;
            const int64_t t0r = bos + (int64_t)local * CH;
            const int64_t rem = eos - t0r;
            const int len = (int)(rem < CH ? rem : CH);
            for (int i = threadIdx.x; i < CH * (BV / 8); i += blockDim.x) {
                const int r = i / (BV / 8), j = i % (BV / 8);
                const bool ok = r < len;
                cp_async16(tn.chunk(r, j), p.dO + ((t0r + (ok ? r : 0)) * p.H + h) * D + col0 + j * 8, ok);
            }
        }
        float* gs = reinterpret_cast<float*>(s + SM::oG);
        const float* gsrc = p.gT + ((size_t)c * p.H + h) * D;
        for (int i = threadIdx.x; i < D / 4; i += blockDim.x) cp_async16(gs + 4 * i, gsrc + 4 * i, true);
        cp_async_commit();
    };

    const int n = ce - cb;
    if (n > 0) issue(role == 0 ? cb : ce - 1, 0);
    for (int it = 0; it < n; ++it) {
        const int c = role == 0 ? cb + it : ce - 1 - it;
        const int b = it & 1;
        unsigned char* s = stage(b);
        TileCD t0{s + SM::oT0}, t1{s + SM::oT1}, t2{s + SM::oT2}, t3{s + SM::oT3};
        TileN tn{s + SM::oN};
        const float* gs = reinterpret_cast<const float*>(s + SM::oG);

        cp_async_wait<0>();
        __syncthreads();
        if (it + 1 < n) issue(role == 0 ? c + 1 : c - 1, b ^ 1);

        // save the state entering this step (S0 of chunk c, or dS_C of chunk c)
        __nv_bfloat16* dst = (role == 0 ? p.S0 : p.dS) + ((size_t)c * p.H + h) * D * D;
        frag_foreach(st, m0, n0, [&](int r, int cc, float a0, float a1) {
            const uint32_t w = pack_bf16(a0, a1);
            *reinterpret_cast<uint32_t*>(sS.ptr(r, cc)) = w;
            dst[(size_t)(col0 + cc) * D + r] = __float2bfloat16(a0);  // saved value-major [dv][dk]
            dst[(size_t)(col0 + cc + 1) * D + r] = __float2bfloat16(a1);
        });
        __syncthreads();

        // role 0: X = W S0 -> Vn = U - X ; role 1: Y = kr dS_C -> -Y
        {
            float x[1][2][4];
            zero_acc(x);
            warp_mma<1, 2, A_ROW, B_ROW>(x, t0, sS, mx, n0, 0, D);
            frag_foreach(x, mx, n0, [&](int r, int cc, float a0, float a1) {
                float o0, o1;
                if (role == 0) {
                    const float2 u = unpack_bf16(*reinterpret_cast<const uint32_t*>(tn.ptr(r, cc)));
                    o0 = u.x - a0;
                    o1 = u.y - a1;
                } else {
                    o0 = -a0;
                    o1 = -a1;
                }
                *reinterpret_cast<uint32_t*>(sY.ptr(r, cc)) = pack_bf16(o0, o1);
            });
        }
        __syncthreads();

        // decay the carried rows, then accumulate the chunk's contribution
        frag_foreach(st, m0, n0, [&](int r, int, float& a0, float& a1) {
            const float gam = __expf(gs[r]);
            a0 *= gam;
            a1 *= gam;
        });
        if (role == 0) {
            warp_mma<MT, 2, A_COL, B_ROW>(st, t1, sY, m0, n0, 0, CH);  // + kr^T Vn
        } else {
            warp_mma<MT, 2, A_COL, B_ROW>(st, t1, tn, m0, n0, 0, CH);  // + R_hi^T dO
            warp_mma<MT, 2, A_COL, B_ROW>(st, t3, tn, m0, n0, 0, CH);  // + R_lo^T dO
            warp_mma<MT, 2, A_COL, B_ROW>(st, t2, sY, m0, n0, 0, CH);  // - W^T Y
        }
    }
    float* out = role == 1 ? p.dh0 : p.ht;  // dh0, or the forward's final state (if asked)
    if (out) {
        const size_t sb = ((size_t)seq * p.H + h) * D * D;
        frag_foreach(st, m0, n0, [&](int r, int c, float a0, float a1) {
            out[sb + (size_t)r * D + col0 + c] = a0;
            out[sb + (size_t)r * D + col0 + c + 1] = a1;
        });
    }
}

template <int D>
static cudaError_t launch_states_t(const Params& p, int role0, int nroles, cudaStream_t s) {
    const int bytes = StateSmem<D>::bytes;
    cudaError_t e = cudaFuncSetAttribute(k_states<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.N * p.H * (D / BV), nroles);
    k_states<D><<<grid, 256, bytes, s>>>(p, role0);
    return cudaGetLastError();
}

cudaError_t launch_states(const Params& p, bool fwd, bool bwd, cudaStream_t s) {
    if (!fwd && !bwd) return cudaSuccess;
    if (p.D == 128) return launch_states_tc(p, fwd, bwd, s);
    const int role0 = fwd ? 0 : 1, nroles = (fwd && bwd) ? 2 : 1;
    return launch_states_t<64>(p, role0, nroles, s);
}

}  // namespace gdr
