// Per-chunk building blocks shared by the chunk-parallel kernels (prep, main).
//
// Gates.  Inside a chunk of C = 64 tokens the cumulative log gate is
// gc[r] = sum_{i<=r} g_i (per channel for KDA), gT = gc[C-1].  The pages'
// derived tiles ("FlashKDA之backward（K1）", forward workspace and §3.2) are
//   kd = kn e^{gc},  ki = kn e^{-gc},  kr = kn e^{gT-gc},  qd = scale qn e^{gc}.
// kd and ki reach e^{+-|gc|} (the page's ~1e20 example), so products inside the
// chunk use tiles referenced to the middle of the chunk's gate range instead:
//   kd' = kn e^{gc-ref}, ki' = kn e^{ref-gc}, qd' = scale qn e^{gc-ref},
// ref = (max gc + min gc) / 2 per channel.  kd' ki'^T = kd ki^T exactly, and
// every factor stays within e^{+-span/2}; a span beyond 160 nats is flagged.
#pragma once
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {

// fp32 gate storage in shared memory
template <int D, bool KDA>
struct Gates {
    static constexpr int LDG = D + 8;  // row stride of gc (KDA)
    float* gc;   // KDA [C][LDG]; GDN [C]
    float* ref;  // KDA [D];      GDN [1]
    float* gT;   // KDA [D];      GDN [1]
    __device__ __forceinline__ float gcv(int r, int d) const { return KDA ? gc[r * LDG + d] : gc[r]; }
    __device__ __forceinline__ float refv(int d) const { return KDA ? ref[d] : ref[0]; }
    __device__ __forceinline__ float gTv(int d) const { return KDA ? gT[d] : gT[0]; }
    static constexpr int floats() { return KDA ? CH * LDG + 2 * D : CH + 2; }
};

// GDN gate of one chunk by the first warp: lane l holds g of rows 2l and 2l + 1 (0 past
// the chunk's end); writes gc (inclusive cumsum), gT and ref = (max gc + min gc) / 2.
template <int D>
__device__ __forceinline__ void gdn_gate_scan(float g0, float g1, const Gates<D, false>& G, bool flag_range,
                                              const Params& p) {
    const int lane = threadIdx.x & 31, r0 = 2 * lane;
    const float s = g0 + g1;
    float incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const float excl = incl - s;
    G.gc[r0] = excl + g0;
    G.gc[r0 + 1] = incl;
    float mx = fmaxf(excl + g0, incl), mn = fminf(excl + g0, incl);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    const float gT = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
        G.gT[0] = gT;
        G.ref[0] = 0.5f * (mx + mn);
        if (flag_range && (0.5f * (mx - mn) > 80.f || mx > 80.f)) atomicOr(p.status, ST_GATE_RANGE);
    }
}

// Computes gc, gT and ref for one (chunk, head).  Rows >= len have g = 0.
// Must be called by every thread of the block (it synchronises); NT = blockDim.x.
template <int D, bool KDA, int NT = 256>
__device__ void load_gates(const Params& p, const ChunkInfo& ci, int h, const Gates<D, KDA>& G,
                           bool flag_range) {
    if constexpr (KDA) {
        // thread = (channel d, segment of RS rows): the raw gates of its rows come from
        // global memory in one batch of independent loads, g = -e^{A_log} softplus(raw +
        // dt_bias) and the inclusive scan run in registers, then the earlier segments'
        // totals (the last row of each segment's local scan) are added as a prefix
        constexpr int NSEG = NT / D, RS = CH / NSEG;
        static_assert(NSEG * D == NT && NSEG * RS == CH, "thread count must tile the C x D gate block");
        const float a = expf(p.A_log[h]);
        const int d = threadIdx.x % D, sg = threadIdx.x / D;
        const float bias = p.dt_bias[h * D + d];
        float v[RS];
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            const int r = sg * RS + i;
            v[i] = r < ci.len ? bf2f(p.g_raw[((ci.t0 + r) * p.H + h) * D + d]) : 0.f;
        }
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < RS; ++i) {
            if (sg * RS + i < ci.len) acc += kda_gate_fn(p.kda_gate, p.gate_scale, a, v[i] + bias);
            v[i] = acc;
        }
        if (sg < NSEG - 1) G.gc[(sg * RS + RS - 1) * G.LDG + d] = acc;
        __syncthreads();
        float pre = 0.f;
        for (int s2 = 0; s2 < sg; ++s2) pre += G.gc[(s2 * RS + RS - 1) * G.LDG + d];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RS; ++i) G.gc[(sg * RS + i) * G.LDG + d] = v[i] + pre;
        __syncthreads();
        for (int dd = threadIdx.x; dd < D; dd += NT) {
            float mx = -3.0e38f, mn = 3.0e38f;
#pragma unroll 16
            for (int r = 0; r < CH; ++r) {
                const float x = G.gc[r * G.LDG + dd];
                mx = fmaxf(mx, x);
                mn = fminf(mn, x);
            }
            G.gT[dd] = G.gc[(CH - 1) * G.LDG + dd];
            G.ref[dd] = 0.5f * (mx + mn);
            if (flag_range && (0.5f * (mx - mn) > 80.f || mx > 80.f)) atomicOr(p.status, ST_GATE_RANGE);
        }
    } else {
        if (threadIdx.x < 32) {
            const int r0 = 2 * threadIdx.x;
            const float g0 = r0 < ci.len ? p.g[(ci.t0 + r0) * p.H + h] : 0.f;
            const float g1 = r0 + 1 < ci.len ? p.g[(ci.t0 + r0 + 1) * p.H + h] : 0.f;
            gdn_gate_scan(g0, g1, G, flag_range, p);
        }
    }
}

// beta = sigmoid(logit) for valid rows, 0 for padding rows.
__device__ __forceinline__ void load_beta(const Params& p, const ChunkInfo& ci, int h, float* sBeta) {
    for (int r = threadIdx.x; r < CH; r += blockDim.x)
        sBeta[r] = r < ci.len ? sigmoid_f(bf2f(p.beta_logit[(ci.t0 + r) * p.H + h])) : 0.f;
}

// Issues cp.async copies of the chunk's rows of a token-major [T,heads,D] tensor
// into a swizzled C x D tile (rows >= len are zero-filled); heads < 0 means p.H.
template <int D, class Tile>
__device__ __forceinline__ void async_load_rows(const Tile& t, const __nv_bfloat16* src, const Params& p,
                                                const ChunkInfo& ci, int h, int heads = -1) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    const int nh = heads < 0 ? p.H : heads;
    for (int i = threadIdx.x; i < CH * CPR; i += blockDim.x) {
        const int r = i / CPR, j = i % CPR;
        const bool ok = r < ci.len;
        const __nv_bfloat16* g = src + ((ci.t0 + (ok ? r : 0)) * nh + h) * D + j * 8;
        cp_async16(t.chunk(r, j), g, ok);
    }
}

// Copies a contiguous tile of ROWS x COLS bf16 (row-major in global memory)
// into a swizzled shared tile.
template <int ROWS, int COLS, class Tile>
__device__ __forceinline__ void async_load_tile(const Tile& t, const __nv_bfloat16* src) {
    constexpr int CPR = COLS / 8;
    for (int i = threadIdx.x; i < ROWS * CPR; i += blockDim.x) {
        const int r = i / CPR, j = i % CPR;
        cp_async16(t.chunk(r, j), src + (int64_t)r * COLS + j * 8, true);
    }
}

// 1/sqrt(sum x^2 + 1e-6) of the 64 rows of a C x D tile (4 threads per row;
// needs blockDim.x >= 256).  Source: shared tile.
template <int D, class Tile>
__device__ __forceinline__ void row_inv_norms_smem(const Tile& t, float* out) {
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    float s = 0.f;
    if (r < CH) {
#pragma unroll
        for (int j = part * (D / 32); j < (part + 1) * (D / 32); ++j) {
            uint4 v = *reinterpret_cast<const uint4*>(t.chunk(r, j));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = unpack_bf16(w[e]);
                s += f.x * f.x + f.y * f.y;
            }
        }
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if (r < CH && part == 0) out[r] = rsqrtf(s + 1e-6f);
}

// Same, reading the chunk's rows of a token-major global tensor.
template <int D>
__device__ __forceinline__ void row_inv_norms_global(const __nv_bfloat16* src, const Params& p,
                                                     const ChunkInfo& ci, int h, float* out, int heads = -1) {
    const int r = threadIdx.x >> 2, part = threadIdx.x & 3;
    float s = 0.f;
    if (r < ci.len) {
        const uint4* g = reinterpret_cast<const uint4*>(src + ((ci.t0 + r) * (heads < 0 ? p.H : heads) + h) * D);
#pragma unroll
        for (int j = part * (D / 32); j < (part + 1) * (D / 32); ++j) {
            uint4 v = g[j];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = unpack_bf16(w[e]);
                s += f.x * f.x + f.y * f.y;
            }
        }
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if (r < CH && part == 0) out[r] = rsqrtf(s + 1e-6f);
}

// Exponent kinds of the derived tiles (factor e^{a gc + b ref + c gT}).
enum Fac { F_KD = 0, F_KDP = 1, F_KIP = 2, F_KR = 3 };  // e^{gc}, e^{gc-ref}, e^{ref-gc}, e^{gT-gc}

template <int KIND, int D, bool KDA>
__device__ __forceinline__ float gate_exponent(const Gates<D, KDA>& G, int r, int d) {
    const float gc = G.gcv(r, d);
    if (KIND == F_KD) return gc;
    if (KIND == F_KDP) return gc - G.refv(d);
    if (KIND == F_KIP) return G.refv(d) - gc;
    return G.gTv(d) - gc;
}

template <int KIND, int D, bool KDA>
__device__ __forceinline__ float gate_factor(const Gates<D, KDA>& G, int r, int d) {
    return __expf(gate_exponent<KIND>(G, r, d));
}

// Element of a derived tile as the tensor cores see it: bf16(x * m * f) with
// m = inv * mul * rowmul.  build_tile and the gate-gradient terms of the main
// kernel both go through these two functions, so they agree bit for bit.
__device__ __forceinline__ float derived_m(float inv, float mul, float rowmul) { return inv * mul * rowmul; }
__device__ __forceinline__ float derived_val(float x, float m, float f) {
    return __bfloat162float(__float2bfloat16_rn(x * m * f));
}

// dst[r][d] = src[r][d] * inv[r] * rowmul[r] * mul * e^{factor KIND}(r, d)
// src: swizzled shared tile (SRC_GLOBAL = false) or the chunk rows of a
// token-major global tensor (SRC_GLOBAL = true).  rowmul may be null.
template <int KIND, int D, bool KDA, bool SRC_GLOBAL, class Tile>
__device__ __forceinline__ void build_tile(const Tile& dst, const Tile& src, const __nv_bfloat16* gsrc,
                                           const Params& p, const ChunkInfo& ci, int h,
                                           const Gates<D, KDA>& G, const float* inv,
                                           const float* rowmul, float mul, const Tile* lo = nullptr,
                                           int heads = -1) {
    // With `lo`, the tile is stored as a bf16 pair: dst = bf16(v), lo = bf16(v - dst).  A
    // global source has `heads` heads per token (heads < 0 means p.H); h indexes them.
    constexpr int CPR = D / 8;
    for (int i = threadIdx.x; i < CH * CPR; i += blockDim.x) {
        const int r = i / CPR, j = i % CPR;
        uint4 v;
        if (SRC_GLOBAL) {
            if (r < ci.len)
                v = *reinterpret_cast<const uint4*>(gsrc + ((ci.t0 + r) * (heads < 0 ? p.H : heads) + h) * D + j * 8);
            else
                v = make_uint4(0, 0, 0, 0);
        } else {
            v = *reinterpret_cast<const uint4*>(src.chunk(r, j));
        }
        const float m = derived_m(inv[r], mul, rowmul ? rowmul[r] : 1.f);
        uint32_t w[4] = {v.x, v.y, v.z, v.w}, wl[4];
        float fr = 0.f;
        if (!KDA) fr = gate_factor<KIND>(G, r, 0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 f = unpack_bf16(w[e]);
            const int d = j * 8 + 2 * e;
            const float f0 = KDA ? gate_factor<KIND>(G, r, d) : fr;
            const float f1 = KDA ? gate_factor<KIND>(G, r, d + 1) : fr;
            const float v0 = f.x * m * f0, v1 = f.y * m * f1;  // == derived_val(x, m, f) once rounded
            w[e] = pack_bf16(v0, v1);
            if (lo) {
                const float2 hv = unpack_bf16(w[e]);
                wl[e] = pack_bf16(v0 - hv.x, v1 - hv.y);
            }
        }
        *reinterpret_cast<uint4*>(dst.chunk(r, j)) = make_uint4(w[0], w[1], w[2], w[3]);
        if (lo) *reinterpret_cast<uint4*>(lo->chunk(r, j)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
}

// Stores two fp32 values at (r, c), (r, c+1) of a bf16 tile, and, with `lo`,
// their bf16 residuals into a second tile.
template <class Tile>
__device__ __forceinline__ void store_pair(const Tile& hi, const Tile* lo, int r, int c, float v0, float v1) {
    const uint32_t w = pack_bf16(v0, v1);
    *reinterpret_cast<uint32_t*>(hi.ptr(r, c)) = w;
    if (lo) {
        const float2 hv = unpack_bf16(w);
        *reinterpret_cast<uint32_t*>(lo->ptr(r, c)) = pack_bf16(v0 - hv.x, v1 - hv.y);
    }
}

// Iterates over the fragment elements of a warp tile, two adjacent columns at a time.
template <int MT, int NT, class F>
__device__ __forceinline__ void frag_foreach(float (&acc)[MT][NT][4], int m0, int n0, F&& f) {
    const int g = frag_g(), c = frag_c();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = m0 + mt * 16 + g + 8 * hf;
                const int col = n0 + nt * 8 + 2 * c;
                f(r, col, acc[mt][nt][2 * hf], acc[mt][nt][2 * hf + 1]);
            }
}

// T = (I + A)^-1 for a strictly lower 64x64 fp32 matrix A (row stride 65).
// Blocked: 16x16 diagonal blocks by forward substitution, then the off-diagonal
// blocks T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj by increasing i - j.
// tmp: 3 * 256 floats.  NT = blockDim.x (a multiple of 256 or 256 exactly); threads
// beyond the first 256 only help clear Tf.  Tf gets the full lower T.
template <int NT = 256>
__device__ inline void invert_unit_lower64(const float* A, float* Tf, float* tmp) {
    constexpr int LD = 65;
    const int t = threadIdx.x;
    for (int i = t; i < 64 * LD; i += NT) Tf[i] = 0.f;
    __syncthreads();
    if (t < 64) {
        const int b = t >> 4, j = t & 15;
        const float* Ab = A + (16 * b) * LD + 16 * b;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < i; ++s) acc -= Ab[i * LD + s] * x[s];
            x[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[(16 * b + i) * LD + 16 * b + j] = x[i];
    }
    __syncthreads();
    for (int L = 1; L < 4; ++L) {
        const int nb = 4 - L;
        for (int e = t; e < nb * 256 && t < 256; e += 256) {
            const int j = e >> 8, i = j + L, r = (e >> 4) & 15, c = e & 15;
            float acc = 0.f;
            for (int k = j; k < i; ++k) {
                const float* Ar = A + (16 * i + r) * LD + 16 * k;
                const float* Tc = Tf + (16 * k) * LD + 16 * j + c;
#pragma unroll
                for (int s = 0; s < 16; ++s) acc += Ar[s] * Tc[s * LD];
            }
            tmp[e] = acc;
        }
        __syncthreads();
        for (int e = t; e < nb * 256 && t < 256; e += 256) {
            const int j = e >> 8, i = j + L, r = (e >> 4) & 15, c = e & 15;
            const float* Tr = Tf + (16 * i + r) * LD + 16 * i;
            const float* M = tmp + (j << 8) + c;
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < 16; ++s) acc += Tr[s] * M[s * 16];
            Tf[(16 * i + r) * LD + 16 * j + c] = -acc;
        }
        __syncthreads();
    }
}

// Warp reductions of the chunk-parallel tcgen05 kernels.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sum over the warp of each of 32 per-lane values: lane l returns the total of v[l]
// (recursive halving: 31 exchanges instead of 32 x 5).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}
// Same for 16 values: lanes l and l ^ 1 return the total of v[l >> 1].
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 2; o >>= 1) {
        const int n = o >> 1;  // values kept after this step
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = up ? v[i] : v[i + n];
            const float keep = up ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

}  // namespace gdr
