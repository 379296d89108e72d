// Shared device helpers for the gated delta-rule kernels (sm_103a).
//
// Conventions used by every kernel in this directory:
//   * chunk length C = 64 tokens; head dim D = dk = dv in {64, 128};
//   * activations are token-major [T_total, H, D] bf16, per-chunk workspace
//     tiles are [chunk][H][rows][cols] contiguous;
//   * shared-memory bf16 tiles are row-major with rows of >= 128 bytes and the
//     16-byte chunks of row r XOR-swizzled by (r & 7), so that ldmatrix of 8
//     consecutive rows is bank-conflict free;
//   * warp-level tensor-core products use mma.sync m16n8k16 bf16 -> fp32.
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

// --------------------------------------------------------------------------
// shared-memory tiles
// --------------------------------------------------------------------------
// Swizzled bf16 tile: ROWB bytes per row (>= 128, multiple of 128).
template <int ROWB>
struct SwzTile {
    static_assert(ROWB % 128 == 0, "swizzled rows must be multiples of 128 bytes");
    unsigned char* base;
    __device__ __forceinline__ uint32_t off(int r, int c) const {  // c: element column
        return r * ROWB + ((((c >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1);
    }
    __device__ __forceinline__ unsigned char* ptr(int r, int c) const { return base + off(r, c); }
    __device__ __forceinline__ uint32_t addr(int r, int c) const { return smem_u32(base) + off(r, c); }
    // 16-byte chunk j of row r (j counts 8-element chunks)
    __device__ __forceinline__ unsigned char* chunk(int r, int j) const {
        return base + r * ROWB + ((j ^ (r & 7)) << 4);
    }
};

// Padded bf16 tile: LDE elements per row (rows of 48 bytes for 16 columns).
template <int LDE>
struct PadTile {
    unsigned char* base;
    __device__ __forceinline__ uint32_t off(int r, int c) const { return (r * LDE + c) * 2; }
    __device__ __forceinline__ unsigned char* ptr(int r, int c) const { return base + off(r, c); }
    __device__ __forceinline__ uint32_t addr(int r, int c) const { return smem_u32(base) + off(r, c); }
    __device__ __forceinline__ unsigned char* chunk(int r, int j) const { return base + (r * LDE + j * 8) * 2; }
};

// --------------------------------------------------------------------------
// ldmatrix / mma.sync
// --------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t a) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Operand storage forms for warp_mma:
//   A_ROW: A stored [M][K] (K contiguous)   A_COL: A stored [K][M] (A^T stored)
//   B_COL: B stored [N][K] (K contiguous)   B_ROW: B stored [K][N] (N contiguous)
enum { A_ROW = 0, A_COL = 1 };
enum { B_COL = 0, B_ROW = 1 };

// acc[MT][NT] (16x8 fp32 fragments) += A[m0.., k0..k0+K) * B[k0.., n0..]
// Rows m0 + 16*mt, columns n0 + 8*nt.  NT must be even.
template <int MT, int NT, int AF, int BF, class TA, class TB>
__device__ __forceinline__ void warp_mma(float (&acc)[MT][NT][4], const TA& A, const TB& B, int m0,
                                         int n0, int k0, int K) {
    static_assert(NT % 2 == 0, "NT must be even");
    const int lane = threadIdx.x & 31;
    const int li = lane >> 3, lj = lane & 7;
#pragma unroll 2
    for (int k = k0; k < k0 + K; k += 16) {
        uint32_t af[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int m = m0 + mt * 16;
            if (AF == A_ROW) {
                ldsm_x4(af[mt], A.addr(m + (lane & 15), k + ((lane >> 4) << 3)));
            } else {
                ldsm_x4_t(af[mt], A.addr(k + ((li >> 1) << 3) + lj, m + ((li & 1) << 3)));
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            const int n = n0 + nt * 8;
            uint32_t bf[4];
            if (BF == B_COL) {
                ldsm_x4(bf, B.addr(n + ((li >> 1) << 3) + lj, k + ((li & 1) << 3)));
            } else {
                ldsm_x4_t(bf, B.addr(k + ((li & 1) << 3) + lj, n + ((li >> 1) << 3)));
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                mma16816(acc[mt][nt], af[mt], bf[0], bf[1]);
                mma16816(acc[mt][nt + 1], af[mt], bf[2], bf[3]);
            }
        }
    }
}

template <int MT, int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[MT][NT][4]) {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
}

// Fragment element coordinates: element e of fragment (mt, nt) of a warp tile
// at (m0, n0) sits at row m0 + 16 mt + g + 8*(e >> 1), column n0 + 8 nt + 2c + (e & 1).
__device__ __forceinline__ int frag_g() { return (threadIdx.x & 31) >> 2; }
__device__ __forceinline__ int frag_c() { return threadIdx.x & 3; }

// --------------------------------------------------------------------------
// cp.async
// --------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
                 "l"(gmem), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

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
__device__ __forceinline__ float kda_gate_fn(int mode, float gs, float a, float x) {
    return mode == 0 ? kda_gate_fn<0>(gs, a, x) : kda_gate_fn<1>(gs, a, x);
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
        const float s = sigmoid_f(a * x);
        const float dz = dgl * (kLn2f * gs) * (s * (1.f - s));
        dA = dz * a * x;
        return dz * a;
    }
}
__device__ __forceinline__ float kda_gate_bwd(int mode, float gs, float a, float x, float dgl, float& dA) {
    return mode == 0 ? kda_gate_bwd<0>(gs, a, x, dgl, dA) : kda_gate_bwd<1>(gs, a, x, dgl, dA);
}

}  // namespace gdr
