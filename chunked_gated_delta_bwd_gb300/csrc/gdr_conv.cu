// Backward of the causal depthwise conv1d (optionally followed by SiLU) that produces q, k
// and v in a gated delta-rule layer ("第三章 反向传播的完整推导", starbuckoverflow.cn, the
// causal-convolution series, chapter 3).  Per channel c, K taps, zero state before each
// sequence's first token:
//
//   z_t = bias_c + sum_k w_{c,k} x_{t-K+1+k},   y = SiLU(z) (or y = z)
//   delta_t = dy_t sigmoid(z_t) (1 + z_t (1 - sigmoid(z_t)))   (or delta = dy)
//   dbias_c = sum_t delta_t,   dw_{c,k} = sum_t delta_t x_{t-K+1+k},
//   dx_s = sum_k w_{c,k} delta_{s+K-1-k}       (delta zero past the sequence end)
//
// The pre-activation z is recomputed from x (not stored by the forward).  HBM-bound: each
// thread owns a pair of consecutive channels (4-byte loads of bf16 x, dy and stores of dx,
// a warp covering 64 contiguous channels, one 128-byte line, of a token row) and walks
// tiles of CONV_TILE tokens in order with the last K - 1 inputs and the last K deltas in
// registers: dx of token s - K + 1 is complete once delta_s is known.  Tiles inside one
// sequence (halos included) take a path without per-token checks whose loads of 16
// consecutive tokens are issued before their arithmetic; tiles at sequence boundaries
// are walked in per-sequence segments.  The arithmetic runs on the channel pair with the
// packed two-lane fp32 instructions.  dw and dbias are accumulated in registers over every
// tile the block visits and added to the outputs with one atomic per (block, channel, tap).
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {

namespace {

constexpr int CONV_TILE = 128;   // tokens per tile
constexpr int CONV_THREADS = 128;
constexpr int CONV_U = 8;        // tokens whose loads are issued together (interior tiles)

__device__ __forceinline__ float2 ld_pair(const uint32_t* p) { return unpack_bf16(__ldg(p)); }

// first token of sequence n (dense layout: N sequences of T / N tokens)
__device__ __forceinline__ int64_t seq_start(const ConvParams& p, int n) {
    return p.cu_seqlens ? p.cu_seqlens[n] : (int64_t)n * (p.T / p.N);
}

// One thread's pair of channels: weights, the running parameter gradients, the last K - 1
// inputs and the last K deltas; the arithmetic on packed two-lane fp32 instructions.
template <int K>
struct ConvLane {
    float2 w[K], bias, dw[K], db, xw[K > 1 ? K - 1 : 1], dl[K];

    // delta_s from x_s, dy_s and the inputs s-K+1 .. s-1 in xw
    __device__ __forceinline__ float2 delta(float2 xs, float2 g, bool silu) const {
        float2 z = __ffma2_rn(w[K - 1], xs, bias);
#pragma unroll
        for (int k = 0; k < K - 1; ++k) z = __ffma2_rn(w[k], xw[k], z);
        if (!silu) return g;
        const float2 sg = make_float2(sigmoid_f(z.x), sigmoid_f(z.y));
        // dy sigmoid(z) (1 + z (1 - sigmoid(z)))
        const float2 u = __ffma2_rn(z, __fadd2_rn(make_float2(1.f, 1.f), make_float2(-sg.x, -sg.y)),
                                    make_float2(1.f, 1.f));
        return __fmul2_rn(__fmul2_rn(g, sg), u);
    }
    // the parameter-gradient terms of an output token s of this thread's tile
    __device__ __forceinline__ void accumulate(float2 d, float2 xs) {
        db = __fadd2_rn(db, d);
        dw[K - 1] = __ffma2_rn(d, xs, dw[K - 1]);
#pragma unroll
        for (int k = 0; k < K - 1; ++k) dw[k] = __ffma2_rn(d, xw[k], dw[k]);
    }
    __device__ __forceinline__ void push(float2 xs, float2 d) {
#pragma unroll
        for (int k = 0; k + 1 < K - 1; ++k) xw[k] = xw[k + 1];
        if (K > 1) xw[K > 1 ? K - 2 : 0] = xs;
#pragma unroll
        for (int k = 0; k + 1 < K; ++k) dl[k] = dl[k + 1];
        dl[K - 1] = d;
    }
    // dx of token s - K + 1 after delta_s was pushed: sum_k w_k delta_{s-k}
    __device__ __forceinline__ uint32_t dx() const {
        float2 o = __fmul2_rn(w[0], dl[K - 1]);
#pragma unroll
        for (int k = 1; k < K; ++k) o = __ffma2_rn(w[k], dl[K - 1 - k], o);
        return pack_bf16(o.x, o.y);
    }
    __device__ __forceinline__ void clear_deltas() {
#pragma unroll
        for (int k = 0; k < K; ++k) dl[k] = make_float2(0.f, 0.f);
    }
};

}  // namespace

template <int K>
__global__ void __launch_bounds__(CONV_THREADS, 8) k_conv1d_bwd(const ConvParams p) {
    const int c0 = (blockIdx.x * CONV_THREADS + threadIdx.x) * 2;  // channels c0, c0 + 1
    if (c0 >= p.C) return;
    const int64_t ch = p.C / 2;  // row stride in channel pairs
    const uint32_t* x2 = reinterpret_cast<const uint32_t*>(p.x) + c0 / 2;
    const uint32_t* g2 = reinterpret_cast<const uint32_t*>(p.dy) + c0 / 2;
    uint32_t* dx2 = reinterpret_cast<uint32_t*>(p.dx) + c0 / 2;
    ConvLane<K> L;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        L.w[k] = make_float2(p.w[c0 * K + k], p.w[(c0 + 1) * K + k]);
        L.dw[k] = make_float2(0.f, 0.f);
    }
    L.bias = p.bias ? make_float2(p.bias[c0], p.bias[c0 + 1]) : make_float2(0.f, 0.f);
    L.db = make_float2(0.f, 0.f);
    const bool silu = p.silu;
    const int64_t ntiles = (p.T + CONV_TILE - 1) / CONV_TILE;
    for (int64_t tile = blockIdx.y; tile < ntiles; tile += gridDim.y) {
        const int64_t t0 = tile * CONV_TILE, t1 = min(t0 + CONV_TILE, p.T);
        // the sequence holding t0: largest n with start(n) <= t0
        int lo = 0, hi = p.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seq_start(p, mid) <= t0) lo = mid;
            else hi = mid - 1;
        }
        int n = lo;
        while (n < p.N - 1 && seq_start(p, n + 1) <= t0) ++n;  // past empty sequences
        if (t1 - t0 == CONV_TILE && t0 >= K - 1 && seq_start(p, n) <= t0 - (K - 1) &&
            t1 + (K - 1) <= seq_start(p, n + 1) && seq_start(p, n + 1) <= p.T) {
            // interior tile: the tile and both halos inside one sequence; no per-token checks
#pragma unroll
            for (int k = 0; k < K - 1; ++k) L.xw[k] = ld_pair(x2 + (t0 - (K - 1) + k) * ch);
            L.clear_deltas();
            const uint32_t* px = x2 + t0 * ch;
            const uint32_t* pg = g2 + t0 * ch;
            uint32_t* pd = dx2 + (t0 - (K - 1)) * ch;  // dx of token s - K + 1
            for (int grp = 0; grp < CONV_TILE / CONV_U; ++grp) {
                uint32_t xr[CONV_U], gr[CONV_U];
#pragma unroll
                for (int i = 0; i < CONV_U; ++i) {
                    xr[i] = __ldg(px);
                    gr[i] = __ldg(pg);
                    px += ch;
                    pg += ch;
                }
#pragma unroll
                for (int i = 0; i < CONV_U; ++i) {
                    const float2 xs = unpack_bf16(xr[i]);
                    const float2 d = L.delta(xs, unpack_bf16(gr[i]), silu);
                    L.accumulate(d, xs);
                    L.push(xs, d);
                    if (grp > 0 || i >= K - 1) *pd = L.dx();  // tokens before t0 belong to the previous tile
                    pd += ch;
                }
            }
#pragma unroll
            for (int j = 0; j < K - 1; ++j) {  // right halo: deltas of the next K - 1 tokens
                const float2 xs = ld_pair(px);
                const float2 d = L.delta(xs, ld_pair(pg), silu);
                L.push(xs, d);
                *pd = L.dx();
                px += ch;
                pg += ch;
                pd += ch;
            }
            continue;
        }
        // edge tile: walk it in segments [a, b) of one sequence each, with per-token checks
        int64_t a = t0;
        while (a < t1) {
            while (n < p.N - 1 && seq_start(p, n + 1) <= a) ++n;  // skip sequences ending at or before a
            // [bos, eos): the sequence of token a (clamped so that inconsistent cu_seqlens
            // still read and write inside the tensors and the walk advances)
            const int64_t bos = seq_start(p, n);
            const int64_t eos = min(max(seq_start(p, n + 1), a + 1), p.T);
            const int64_t b = min(t1, eos);  // segment [a, b)
#pragma unroll
            for (int k = 0; k < K - 1; ++k) {
                const int64_t s = a - (K - 1) + k;
                L.xw[k] = (s >= bos && s >= 0) ? ld_pair(x2 + s * ch) : make_float2(0.f, 0.f);
            }
            L.clear_deltas();
            for (int64_t s = a; s < b + K - 1; ++s) {
                float2 d = make_float2(0.f, 0.f);  // past the sequence end: zero
                float2 xs = make_float2(0.f, 0.f);
                if (s < eos) {
                    xs = ld_pair(x2 + s * ch);
                    d = L.delta(xs, ld_pair(g2 + s * ch), silu);
                    if (s < b) L.accumulate(d, xs);
                }
                L.push(xs, d);
                if (s - (K - 1) >= a) dx2[(s - (K - 1)) * ch] = L.dx();
            }
            a = b;
        }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        atomicAdd(&p.dw[c0 * K + k], L.dw[k].x);
        atomicAdd(&p.dw[(c0 + 1) * K + k], L.dw[k].y);
    }
    if (p.dbias) {
        atomicAdd(&p.dbias[c0], L.db.x);
        atomicAdd(&p.dbias[c0 + 1], L.db.y);
    }
}

template <int K>
static cudaError_t launch_conv1d_bwd_t(const ConvParams& p, cudaStream_t s) {
    // one wave: as many blocks as fit on the SMs at once (the blocks loop over token tiles)
    const int gx = (p.C / 2 + CONV_THREADS - 1) / CONV_THREADS;
    const int64_t ntiles = (p.T + CONV_TILE - 1) / CONV_TILE;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_conv1d_bwd<K>, CONV_THREADS, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t gy = (int64_t)per_sm * num_sms() / gx;
    if (gy < 1) gy = 1;
    if (gy > ntiles) gy = ntiles;
    if (gy > 65535) gy = 65535;
    k_conv1d_bwd<K><<<dim3(gx, (unsigned)gy), CONV_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_conv1d_bwd(const ConvParams& p, cudaStream_t s) {
    if (p.T == 0) return cudaSuccess;
    switch (p.K) {
        case 1: return launch_conv1d_bwd_t<1>(p, s);
        case 2: return launch_conv1d_bwd_t<2>(p, s);
        case 3: return launch_conv1d_bwd_t<3>(p, s);
        case 4: return launch_conv1d_bwd_t<4>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdr
