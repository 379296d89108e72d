// Triangular inverse of the chunk algebra, T = (I + A)^-1 for a strictly lower 64 x 64
// fp32 A, on warp-level tf32 tensor-core instructions in a three-term split (fp32
// accuracy): the 16 x 16 diagonal blocks by forward substitution (one thread per column),
// then every 8-column strip of the block rows below its diagonal block by block forward
// substitution T_i = -T_ii sum_k A_ik T_k.  The shapes are below tcgen05's minimum M.
// Shared by the chunk-parallel preparation kernels of both gate kinds.
#pragma once
#include "gdr_common.cuh"
#include "gdr_tc.cuh"

namespace gdr {
namespace inv {

constexpr int LDF = 68;  // row stride of the fp32 64 x 64 matrices of the inversion
constexpr int XLD = 20;  // row stride of a warp's 16 x 8 transfer tile (stored [col][row])

// tf32 split of an fp32 value: hi keeps the top 10 mantissa bits, lo the rest (the tensor
// cores read the top 19 bits of each operand register)
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}
// d += a b for a 16 x 8 (k) A fragment and an 8 (k) x 8 B fragment, tf32 in, fp32 out
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// d += a b to fp32 accuracy: three accumulators for hi hi, hi lo and lo hi
__device__ __forceinline__ void mma_3xtf32(float (&d)[3][4], const float (&a)[4], const float (&b)[2]) {
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
#pragma unroll
    for (int i = 0; i < 2; ++i) split_tf32(b[i], bh[i], bl[i]);
    mma_tf32(d[0], ah, bh);
    mma_tf32(d[1], ah, bl);
    mma_tf32(d[2], al, bh);
}

// Block rows JB+1 .. 3 of the 8-column strip n0 of T (one warp), given the diagonal blocks:
// T_i = -T_ii M_i, M_i = sum_{k=JB}^{i-1} A_ik T_k; every loop has compile-time bounds so
// that the operand loads of a product are issued together.
template <int JB>
__device__ __forceinline__ void invert_strip(const float* sA, float* tT, float* xf, unsigned char* sT,
                                             __nv_bfloat16* gT, int n0, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int i = JB + 1; i < 4; ++i) {
        float acc[3][4] = {};
#pragma unroll
        for (int k = JB; k < i; ++k) {  // M = sum_k A_ik T_k
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int kk = 16 * k + 8 * ks;
                const float* Ar = sA + (16 * i + gid) * LDF + kk + tig;
                const float* Br = tT + (n0 + gid) * LDF + kk + tig;
                const float a[4] = {Ar[0], Ar[8 * LDF], Ar[4], Ar[8 * LDF + 4]};
                const float bb[2] = {Br[0], Br[4]};
                mma_3xtf32(acc, a, bb);
            }
        }
        // M (accumulator layout: rows gid, gid + 8; columns 2 tig, 2 tig + 1) -> xf[col][row]
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float mval = acc[0][e] + (acc[1][e] + acc[2][e]);
            xf[(2 * tig + (e & 1)) * XLD + gid + 8 * (e >> 1)] = mval;
        }
        __syncwarp();
        float out[3][4] = {};
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {  // T_i = -T_ii M
            const int cc = 16 * i + 8 * ks + tig, rr = 16 * i + gid;
            const float a[4] = {tT[cc * LDF + rr], tT[cc * LDF + rr + 8], tT[(cc + 4) * LDF + rr],
                                tT[(cc + 4) * LDF + rr + 8]};
            const float bb[2] = {xf[gid * XLD + 8 * ks + tig], xf[gid * XLD + 8 * ks + tig + 4]};
            mma_3xtf32(out, a, bb);
        }
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            t[e] = -(out[0][e] + (out[1][e] + out[2][e]));
            tT[(n0 + 2 * tig + (e & 1)) * LDF + 16 * i + gid + 8 * (e >> 1)] = t[e];
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int r = 16 * i + gid + 8 * h2, c = n0 + 2 * tig;
            const uint32_t w = pack_bf16(t[2 * h2], t[2 * h2 + 1]);
            *reinterpret_cast<uint32_t*>(sT + tc::sw_off(r, c, 64)) = w;
            if (gT) *reinterpret_cast<uint32_t*>(gT + r * CH + c) = w;
        }
        __syncwarp();
    }
}

// T = (I + A)^-1 for a strictly lower 64 x 64 fp32 A (row-major, stride LDF), by warps 0-7
// (the first 256 threads; named barrier 1).  Writes T in fp32 transposed (tT[c][r], the
// operand copy), and in bf16 [r][c] into the swizzled tile sT and (unless gT is null) the
// global tile gT; the blocks above the diagonal are not written.
__device__ __forceinline__ void invert_tc(const float* sA, float* tT, float* xfer, unsigned char* sT,
                                          __nv_bfloat16* gT) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < 64) {  // diagonal block b, column j: forward substitution down the block
        const int b = tid >> 4, j = tid & 15;
        const float* Ab = sA + 16 * b * LDF + 16 * b;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a[16];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (4 * q < i) {
                    const float4 v = *reinterpret_cast<const float4*>(Ab + i * LDF + 4 * q);
                    a[4 * q] = v.x;
                    a[4 * q + 1] = v.y;
                    a[4 * q + 2] = v.z;
                    a[4 * q + 3] = v.w;
                }
            float acc = i == j ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < i; ++s) acc = fmaf(-a[s], x[s], acc);
            x[i] = acc;
        }
        float* dst = tT + (16 * b + j) * LDF + 16 * b;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * b + i, c = 16 * b + j;
            const __nv_bfloat16 y = __float2bfloat16(x[i]);
            *reinterpret_cast<__nv_bfloat16*>(sT + tc::sw_off(r, c, 64)) = y;
            if (gT) gT[r * CH + c] = y;
        }
    }
    tc::named_sync(1, 256);
    // strip of columns n0 .. n0+7 (block column jb), block rows jb+1 .. 3
    const int n0 = 8 * warp, jb = warp >> 1;
    float* xf = xfer + warp * 8 * XLD;
    switch (jb) {
        case 0: invert_strip<0>(sA, tT, xf, sT, gT, n0, lane); break;
        case 1: invert_strip<1>(sA, tT, xf, sT, gT, n0, lane); break;
        case 2: invert_strip<2>(sA, tT, xf, sT, gT, n0, lane); break;
        default: break;
    }
}

}  // namespace inv
}  // namespace gdr
