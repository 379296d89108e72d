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

// fp32 storage in shared memory of the scalar (GDN) gate of one chunk: the inclusive cumsum
// gc[r], ref = (max gc + min gc) / 2 and gT = gc[C-1]
struct ScalarGates {
    float* gc;   // [C]
    float* ref;  // [1]
    float* gT;   // [1]
    __device__ __forceinline__ float gcv(int r) const { return gc[r]; }
    __device__ __forceinline__ float refv() const { return ref[0]; }
    __device__ __forceinline__ float gTv() const { return gT[0]; }
};

// GDN gate of one chunk by the first warp: lane l holds g of rows 2l and 2l + 1 (0 past
// the chunk's end); writes gc (inclusive cumsum), gT and ref = (max gc + min gc) / 2.
__device__ __forceinline__ void gdn_gate_scan(float g0, float g1, const ScalarGates& G, bool flag_range,
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

// Exponent kinds of the derived tiles (factor e^{a gc + b ref + c gT}).
enum Fac { F_KD = 0, F_KDP = 1, F_KIP = 2, F_KR = 3 };  // e^{gc}, e^{gc-ref}, e^{ref-gc}, e^{gT-gc}

template <int KIND>
__device__ __forceinline__ float gate_exponent(const ScalarGates& G, int r) {
    const float gc = G.gcv(r);
    if (KIND == F_KD) return gc;
    if (KIND == F_KDP) return gc - G.refv();
    if (KIND == F_KIP) return G.refv() - gc;
    return G.gTv() - gc;
}

template <int KIND>
__device__ __forceinline__ float gate_factor(const ScalarGates& G, int r) {
    return __expf(gate_exponent<KIND>(G, r));
}

// Row factor of a derived tile element as the tensor cores see it: bf16(x * m * f) with
// m = inv * mul * rowmul (the prep and main kernels build their tiles and the main
// kernel its gate-gradient terms from the same m, so they agree bit for bit).
__device__ __forceinline__ float derived_m(float inv, float mul, float rowmul) { return inv * mul * rowmul; }

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
