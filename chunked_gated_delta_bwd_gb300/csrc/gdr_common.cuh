// Shared device helpers for the gated delta-rule kernels (sm_103a).
//
// Conventions used by every kernel in this directory:
//   * chunk length C = 64 tokens; the kernels run on D = dk = dv = 128 channels
//     (head_dim 64 reaches them zero-padded to 128);
//   * activations are token-major [T_total, H, D] bf16, per-chunk workspace
//     tiles are [chunk][H][rows][cols] contiguous;
//   * shared-memory operand tiles use the 128-byte swizzle of the tensor-core
//     descriptors (gdr_tc.cuh).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

constexpr int CH = 64;  // chunk length

// Status bits OR-ed into the workspace status word by device code.
constexpr int ST_BAD_SEQLENS = 1;  // cu_seqlens not monotone / wrong total
constexpr int ST_GATE_RANGE = 2;   // a chunk's gate span exceeds the exponent range handled
constexpr int ST_MMA_TIMEOUT = 4;  // a bounded wait for the tensor cores ran out (the CTA gave up)
constexpr int ST_STATES_MISMATCH = 8;  // the states buffer was written for another variant or shape

// --------------------------------------------------------------------------
// small utilities
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Elements i, i + 1 of a register array as a pair for the two-wide fp32 instructions
// (__fmul2_rn, __fadd2_rn, __ffma2_rn), and a pair written back.
#define F2(a, i) make_float2((a)[i], (a)[(i) + 1])
#define ACC2(a, i, expr)            \
    do {                            \
        const float2 r_ = (expr);   \
        (a)[i] = r_.x;              \
        (a)[(i) + 1] = r_.y;        \
    } while (0)

// --------------------------------------------------------------------------
// chunk table lookup
// --------------------------------------------------------------------------
struct ChunkInfo {
    int seq;     // sequence index
    int64_t t0;  // first token of the chunk (global token index)
    int len;     // valid rows (1..64)
    int local;   // chunk index within the sequence
};

// chunk_off: int32 [N+1] prefix sums of per-sequence chunk counts (device), or
// nullptr for the dense layout (N sequences of seq_len tokens each).
__device__ __forceinline__ bool lookup_chunk(int gc, int N, const int* chunk_off,
                                             const int64_t* cu_seqlens, int64_t seq_len,
                                             ChunkInfo& ci) {
    if (chunk_off == nullptr) {
        const int per = (int)((seq_len + CH - 1) / CH);
        if (per == 0 || gc >= per * N) return false;
        ci.seq = gc / per;
        ci.local = gc - ci.seq * per;
        ci.t0 = (int64_t)ci.seq * seq_len + (int64_t)ci.local * CH;
        { const int64_t rem = seq_len - (int64_t)ci.local * CH; ci.len = (int)(rem < CH ? rem : CH); }
        return true;
    }
    if (gc >= chunk_off[N]) return false;
    int lo = 0, hi = N - 1;  // largest s with chunk_off[s] <= gc
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
    }
    ci.seq = lo;
    ci.local = gc - chunk_off[lo];
    const int64_t bos = cu_seqlens[lo], eos = cu_seqlens[lo + 1];
    ci.t0 = bos + (int64_t)ci.local * CH;
    { const int64_t rem = eos - ci.t0; ci.len = (int)(rem < CH ? rem : CH); }
    return true;
}

// softplus(x) = max(x, 0) + log(1 + e^{-|x|}).  With y = e^{-|x|} in (0, 1]:
// y >= 1/16 takes the hardware logarithm of 1 + y (absolute error ~1e-7 on a
// result >= 0.06); smaller y takes the alternating series of log(1 + y) to y^6
// (truncation below 1e-9 relative).  Relative error of the result ~3e-6.
__device__ __forceinline__ float softplus_f(float x) {
    const float y = __expf(-fabsf(x));
    float l;
    if (y >= 0.0625f) {
        l = __logf(1.f + y);
    } else {
        l = y * (1.f - y * (0.5f - y * (1.f / 3.f - y * (0.25f - y * (0.2f - y * (1.f / 6.f))))));
    }
    return fmaxf(x, 0.f) + l;
}
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
// softplus(x) (as softplus_f) and sigmoid(x) from one exponential y = e^{-|x|}:
// sigmoid = 1 / (1 + y) for x >= 0, y / (1 + y) otherwise.
__device__ __forceinline__ void softplus_sigmoid(float x, float& sp, float& sg) {
    const float y = __expf(-fabsf(x));
    float l;
    if (y >= 0.0625f) {
        l = __logf(1.f + y);
    } else {
        l = y * (1.f - y * (0.5f - y * (1.f / 3.f - y * (0.25f - y * (0.2f - y * (1.f / 6.f))))));
    }
    sp = fmaxf(x, 0.f) + l;
    const float inv = __fdividef(1.f, 1.f + y);
    sg = x >= 0.f ? inv : y * inv;
}

// KDA per-channel log gate of one element, x = g_raw + dt_bias, a = e^{A_log}:
//   mode 0 (softplus):         g = -a softplus(x)
//   mode 1 (sigmoid-bounded):  g = ln2 gs sigmoid(a x)  ("FlashKDA之backward（K1）" §5.2: the
//                              base-2 log gate gs sigmoid(a x), written in natural log)
constexpr float kLn2f = 0.6931471805599453f;
template <int MODE>
__device__ __forceinline__ float kda_gate_fn(float gs, float a, float x) {
    if constexpr (MODE == 0) return -a * softplus_f(x);
    else return kLn2f * gs * sigmoid_f(a * x);
}
// Its chain rule for one element: dgl = dL/dg.  Returns dL/dg_raw (which is also the
// element's dt_bias term) and sets dA, the element's term of dL/dA_log.
//   mode 0: dg/dx = -a sigmoid(x), dg/dA_log = g
//   mode 1: dg/dz = ln2 gs s (1 - s) with z = a x, s = sigmoid(z); dz/dx = a, dz/dA_log = a x
template <int MODE>
__device__ __forceinline__ float kda_gate_bwd(float gs, float a, float x, float dgl, float& dA) {
    if constexpr (MODE == 0) {
        float sp, sg;
        softplus_sigmoid(x, sp, sg);
        dA = dgl * (-a * sp);
        return dgl * (-a * sg);
    } else {
        // s (1 - s) from one exponential y = e^{-|z|}: s and 1 - s are 1 / (1 + y) and
        // y / (1 + y) (in the order of the sign of z), neither formed by a cancelling subtraction
        const float z = a * x, y = __expf(-fabsf(z)), inv = __fdividef(1.f, 1.f + y);
        const float dz = dgl * (kLn2f * gs) * (y * inv * inv);
        dA = dz * z;
        return dz * a;
    }
}

}  // namespace gdr
