// Forward output of every chunk, chunk-parallel, from the chunk-start states and the
// prep tiles:
//
//   o = qd S0 + P u,  u = U - W S0    =>    o = (qd - P W) S0 + P U = R S0 + P U
//
// (the chunked forward of "FlashKDA之backward（K1）" §0.1, whose o is the starting point
// of the backward; qd carries the output scale; R is the same tile the state-gradient
// recurrence reads, the X/R form of the FlashQLA GDN backward page, §三).  Rows past a
// sequence's end are not written.
//
// D = 128: one CTA of 4 warps per (chunk, head), several CTAs per SM.  S0 (value-major
// [dv][dk]), R^T and U^T (channel-major [D][C]) and P ([C][C]) arrive by TMA; the
// product o^T = S0^T R^T + U^T P^T (M = 128 value channels) runs on tcgen05 into 64
// tensor-memory columns; thread = value channel, 64 token rows.  (head_dim 64 runs on
// the channels zero-padded to 128.)
#include "gdr_chunk.cuh"
#include "gdr_tc.cuh"
#include "gdr_tma.h"

namespace gdr {

namespace {

constexpr int OD = 128;
constexpr int oS0 = 0;          // S0^T [dv][dk], two 64-column blocks (32 KB)
constexpr int oR = 32768;       // R^T [dk][C] (16 KB)
constexpr int oU = 49152;       // U^T [dv][C] (16 KB)
constexpr int oP = 65536;       // P [r][s] (8 KB)
constexpr int oBar = 73728;     // two mbarriers, the tensor-memory slot
constexpr int OUT_SMEM = oBar + 64 + 1024;
constexpr int LOAD_BYTES = 32768 + 16384 + 16384 + 8192;

struct OutMaps {
    CUtensorMap S0, R, U, P;
};

}  // namespace

__global__ void __launch_bounds__(128) k_out_tc(const Params p, const __grid_constant__ OutMaps m) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x, chunk = item / p.H, h = item % p.H;
    ChunkInfo ci;
    if (!lookup_chunk(chunk, p.N, p.chunk_off, p.cu_seqlens, p.seq_len, ci)) return;  // past the last chunk

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + oBar);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
    const uint32_t mload = smem_u32(bars), mb = smem_u32(bars + 1);
    if (warp == 0) tc::alloc(smem_u32(tslot), 64);
    if (tid == 0) {
        tc::mbar_init(mload, 1);
        tc::mbar_init(mb, 1);
        const int rdd = item * OD;  // 128-row tiles of the chunk-head
        tc::mbar_expect_tx(mload, LOAD_BYTES);
        tc::tma_load_3d(sb + oS0, &m.S0, 0, rdd, 0, mload);
        tc::tma_load_2d(sb + oR, &m.R, 0, rdd, mload);
        tc::tma_load_2d(sb + oU, &m.U, 0, rdd, mload);
        tc::tma_load_2d(sb + oP, &m.P, 0, item * CH, mload);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    // Bounded waits: on a timeout the status word records it and the CTA skips the rest,
    // after a second bounded wait for the copies or products still in flight.
    bool ok = tc::mbar_wait(mload, 0);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicOr(p.status, ST_MMA_TIMEOUT);
    } else {
        if (tid == 0) {
            tc::fence_after();
            constexpr uint32_t id_r = tc::idesc(128, 64, 0, 1), id_p = tc::idesc(128, 64, 0, 0);
#pragma unroll
            for (int k = 0; k < OD; k += 16)  // o^T = S0^T R^T
                tc::mma(tmem, tc::kdesc(sb + oS0, OD, 0, k), tc::mdesc(sb + oR, OD, 0, k), id_r, k > 0);
#pragma unroll
            for (int k = 0; k < CH; k += 16)  // + U^T P^T
                tc::mma(tmem, tc::kdesc(sb + oU, OD, 0, k), tc::kdesc(sb + oP, CH, 0, k), id_p, 1);
            tc::commit(mb);
        }
        ok = tc::mbar_wait(mb, 0);
        tc::fence_after();
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(p.status, ST_MMA_TIMEOUT);
                tc::mbar_wait(mb, 0);
            }
        } else {
            // thread = value channel L (tensor-memory lane), columns = the chunk's rows
            const int L = 32 * warp + lane;
            __nv_bfloat16* dst = p.o + (ci.t0 * p.H + h) * OD + L;
            const int64_t rs = (int64_t)p.H * OD;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tc::ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * half, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int r = 32 * half + i;
                    if (r < ci.len) dst[r * rs] = __float2bfloat16(v[i]);
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, 64);
}

cudaError_t launch_out(const Params& p, cudaStream_t s) {
    const int items = p.max_chunks * p.H;
    if (items == 0) return cudaSuccess;
    if (p.D != OD) return cudaErrorInvalidValue;  // (head_dim 64 runs zero-padded to 128)
    OutMaps m;
    const uint64_t rows_dd = (uint64_t)p.max_chunks * p.H * OD;
    const uint64_t rows_cc = (uint64_t)p.max_chunks * p.H * CH;
    if (!(encode_blocked_rows_map(&m.S0, p.S0, rows_dd, OD) && encode_rows_map(&m.R, p.R, rows_dd, CH, OD) &&
          encode_rows_map(&m.U, p.U, rows_dd, CH, OD) && encode_rows_map(&m.P, p.Pm, rows_cc, CH, CH)))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, OUT_SMEM);
    if (e != cudaSuccess) return e;
    k_out_tc<<<items, 128, OUT_SMEM, s>>>(p, m);
    return cudaGetLastError();
}

}  // namespace gdr
