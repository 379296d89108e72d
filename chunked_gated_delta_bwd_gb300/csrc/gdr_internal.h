// Internal launch parameters shared by the host launcher and the kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdr {

struct Params {
    // shape
    int N, H, D;
    int Hk;                 // q / k heads (GQA: H is a multiple; value head h reads q / k head h / (H / Hk))
    __nv_bfloat16 *dq_out, *dk_out;  // GQA: the caller's dq / dk [T,Hk,D] (dq / dk hold per-value-head terms)
    int64_t T_total;
    int64_t seq_len;        // dense layout: tokens per sequence (T_total / N)
    int max_chunks;         // upper bound on the number of chunks (grid size)
    const int64_t* cu_seqlens;  // device [N+1] or nullptr (dense)
    const int* chunk_off;   // device [N+1] chunk prefix sums, or nullptr (dense)
    float scale;
    int kda;                // 0: scalar GDN gate, 1: per-channel KDA gate
    int kda_gate;           // KDA gate function: 0 softplus, 1 sigmoid-bounded (gdr.h)
    float gate_scale;       // sigmoid-bounded gate: g = ln2 gate_scale sigmoid(e^{A_log} x)

    // inputs
    const __nv_bfloat16 *q, *k, *v, *dO, *beta_logit;
    const float* g;                 // GDN log gate [T,H]
    const __nv_bfloat16* g_raw;     // KDA raw gate [T,H,D]
    const float *A_log, *dt_bias;   // KDA [H], [H,D]
    const float *h0, *dht;          // [N,H,D,D] or nullptr

    // workspace
    int* status;
    // per chunk-head tiles: W, U, Kr, R, Rlo [C][D] (D = 64) or channel-major [D][C]
    // (D = 128, the layout the tcgen05 state recurrence reads); T [C][C]
    __nv_bfloat16 *W, *U, *Kr, *R, *Rlo, *Tm;
    __nv_bfloat16* Pm;                   // forward only: P = lower(qd ki^T) [C][C] per chunk-head, or nullptr
    // KDA backward only: the in-chunk matrices of the prep kernel's first product for the main
    // kernel, [3][C][C] bf16 per chunk-head: A = strict_lower(diag(beta) A_raw), then P as a
    // bf16 pair (hi, lo); or nullptr
    __nv_bfloat16* APm;
    float *gT, *egT;                     // [chunk][H][D]: chunk gate total and its exponential
    __nv_bfloat16 *S0, *dS;              // per chunk-head states, value-major [dv][dk]
    // time-parallel state passing (seg_G > 1): per (sequence, head) and segment, fp32 key-major
    // [D][D]: segment results from zero (role 0 / role 1), segment transitions, segment starts.
    // seg_G serves calls that run both state directions, seg_G1 calls that run one; the
    // kernels read seg_G, which the state launcher sets to the count of the call
    int seg_G, seg_G1;
    float *segL, *segLb, *segP, *segS;

    // saved chunk states (a backward from the buffer of a forward call): the buffer's header,
    // which the main kernels compare with the header this call expects, or nullptr
    const int* states_hdr;
    int states_tag[16];
    int test_stall;                 // test hook: main-kernel CTA index + 1 held at its first item (0: none)

    // outputs
    __nv_bfloat16* o;               // forward output [T,H,D]
    float* ht;                      // forward final state [N,H,D,D] (key-major), or nullptr
    __nv_bfloat16 *dq, *dk, *dv, *dbeta;
    float* dg;                      // GDN [T,H]
    __nv_bfloat16* dg_raw;          // KDA [T,H,D]
    float *dh0, *dA_log, *ddt_bias;
};

// q / k head of value head h
__host__ __device__ __forceinline__ int qk_head(const Params& p, int h) { return h / (p.H / p.Hk); }

#ifdef __CUDACC__
// The saved states' header matches this call (or the states are recomputed inside the call).
// Every thread of a CTA reads the same 16 words, so the answer is uniform over the CTA.
__device__ __forceinline__ bool states_header_ok(const Params& p) {
    if (!p.states_hdr) return true;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 16; ++i) ok &= __ldg(p.states_hdr + i) == p.states_tag[i];
    return ok;
}
#endif

// multiprocessors of the current device (cached per device)
inline int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

// causal depthwise conv1d backward (gdr_conv1d_bwd)
struct ConvParams {
    int N;                        // sequences
    int64_t T;                    // tokens
    int C, K, silu;               // channels, taps, SiLU after the conv
    const int64_t* cu_seqlens;    // device [N+1] or nullptr (dense)
    const __nv_bfloat16 *x, *dy;  // [T][C]
    const float *w, *bias;        // [C][K], [C] or nullptr
    __nv_bfloat16* dx;            // [T][C]
    float *dw, *dbias;            // [C][K], [C] or nullptr (accumulated: zeroed by the caller)
};
cudaError_t launch_conv1d_bwd(const ConvParams& p, cudaStream_t s);

cudaError_t launch_chunk_table(const Params& p, cudaStream_t s);
cudaError_t launch_prep(const Params& p, cudaStream_t s);
cudaError_t launch_prep_kda(const Params& p, cudaStream_t s);  // KDA, D = 128, tcgen05 + TMA
cudaError_t launch_prep_gdn(const Params& p, cudaStream_t s);  // GDN, D = 128, tcgen05 + TMA on the raw q, k tiles
cudaError_t launch_states(const Params& p, bool fwd, bool bwd, cudaStream_t s);
cudaError_t launch_states_tc(const Params& p, bool fwd, bool bwd, cudaStream_t s);  // D = 128, tcgen05 + TMA
int states_kernel_count(const Params& p, bool fwd, bool bwd);  // kernels launch_states_tc launches
cudaError_t launch_main(const Params& p, cudaStream_t s);
cudaError_t launch_main_kda(const Params& p, cudaStream_t s);  // KDA, D = 128, tcgen05 + TMA
cudaError_t launch_main_gdn(const Params& p, cudaStream_t s);  // GDN, D = 128, tcgen05 + TMA on the raw q, k tiles
cudaError_t launch_out(const Params& p, cudaStream_t s);       // forward output o = R S0 + P U
cudaError_t launch_group_sum(const Params& p, cudaStream_t s);  // GQA: dq, dk summed over each head group

}  // namespace gdr
