// C ABI of the library (declared in include/gdr.h): argument checks, the
// workspace layout, the varlen chunk table and the launch sequence.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/gdr.h"
#include "gdr_common.cuh"
#include "gdr_internal.h"

namespace gdr {

static thread_local char g_err[512] = "";

static gdr_status fail(gdr_status s, const char* fmt, const char* what = "") {
    snprintf(g_err, sizeof(g_err), fmt, what);
    return s;
}

static gdr_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_err, sizeof(g_err), "%s: %s", where, cudaGetErrorString(e));
    return GDR_ERR_CUDA;
}

// chunk_off[s] = sum_{i<s} ceil(len_i / 64); validates cu_seqlens on the device.
// One CTA of 1024 threads; thread t owns a contiguous range of sequences.
__global__ void __launch_bounds__(1024) k_chunk_table(const int64_t* cu, int N, int64_t T, int* chunk_off,
                                                      int* status) {
    __shared__ int s_tot[1024];
    __shared__ int s_bad;
    const int t = threadIdx.x;
    if (t == 0) s_bad = 0;
    __syncthreads();
    const int per = (N + 1023) / 1024;
    const int a = min(N, t * per), b = min(N, a + per);
    int cnt = 0;
    bool bad = false;
    for (int s = a; s < b; ++s) {
        const int64_t l = cu[s + 1] - cu[s];
        if (l < 0) bad = true;
        else cnt += (int)((l + CH - 1) / CH);
    }
    if (t == 0 && (cu[0] != 0 || cu[N] != T)) bad = true;
    if (bad) atomicOr(&s_bad, 1);
    s_tot[t] = cnt;
    __syncthreads();
    // inclusive scan of the per-thread totals (Hillis-Steele)
    for (int o = 1; o < 1024; o <<= 1) {
        const int v = t >= o ? s_tot[t - o] : 0;
        __syncthreads();
        s_tot[t] += v;
        __syncthreads();
    }
    if (s_bad) {
        for (int s = t; s <= N; s += 1024) chunk_off[s] = 0;
        if (t == 0) atomicOr(status, ST_BAD_SEQLENS);
        return;
    }
    int run = s_tot[t] - cnt;
    for (int s = a; s < b; ++s) {
        chunk_off[s] = run;
        run += (int)((cu[s + 1] - cu[s] + CH - 1) / CH);
    }
    if (t == 1023) chunk_off[N] = s_tot[1023];
}

// GQA: dq and dk of each q / k head are the sums of the terms of its value heads
// (bf16 [T][H][D] in the workspace, summed in fp32); eight channels per thread, both tensors.
__global__ void __launch_bounds__(256) k_group_sum(const __nv_bfloat16* __restrict__ pq,
                                                   const __nv_bfloat16* __restrict__ pk, __nv_bfloat16* oq,
                                                   __nv_bfloat16* ok, int64_t T, int H, int Hk, int D) {
    const int r = H / Hk;
    const int64_t n8 = T * Hk * D / 8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < 2 * n8; i += (int64_t)gridDim.x * blockDim.x) {
        const bool second = i >= n8;
        const int64_t e = (second ? i - n8 : i) * 8;
        const int64_t t = e / ((int64_t)Hk * D);
        const int rem = (int)(e % ((int64_t)Hk * D)), hk = rem / D, d = rem % D;
        const __nv_bfloat16* src = (second ? pk : pq) + ((t * H + (int64_t)hk * r) * D + d);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < r; ++j) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + (int64_t)j * D);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = unpack_bf16(w[q]);
                acc[2 * q] += f.x;
                acc[2 * q + 1] += f.y;
            }
        }
        uint4 o;
        o.x = pack_bf16(acc[0], acc[1]);
        o.y = pack_bf16(acc[2], acc[3]);
        o.z = pack_bf16(acc[4], acc[5]);
        o.w = pack_bf16(acc[6], acc[7]);
        *reinterpret_cast<uint4*>((second ? ok : oq) + e) = o;
    }
}

cudaError_t launch_group_sum(const Params& p, cudaStream_t s) {
    if (p.T_total == 0) return cudaSuccess;
    k_group_sum<<<8 * num_sms(), 256, 0, s>>>(p.dq, p.dk, p.dq_out, p.dk_out, p.T_total, p.H, p.Hk, p.D);
    return cudaGetLastError();
}

// The header of a saved-states buffer: what the states were computed for.
struct StatesTag {
    int v[16];
};
static StatesTag states_tag(const gdr_shape* sh, int kda, const float* h0, int64_t max_chunks, int orig_dim) {
    StatesTag t;
    memset(&t, 0, sizeof(t));
    t.v[0] = 0x53524447;  // "GDRS"
    t.v[1] = 1;           // header version
    t.v[2] = kda ? 1 + sh->kda_gate : 0;
    t.v[3] = sh->num_seqs;
    t.v[4] = sh->num_heads;
    t.v[5] = sh->num_k_heads > 0 ? sh->num_k_heads : sh->num_heads;
    t.v[6] = sh->head_dim;
    t.v[7] = (int)(sh->total_tokens & 0xffffffff);
    t.v[8] = (int)(sh->total_tokens >> 32);
    t.v[9] = (int)max_chunks;
    if (kda && sh->kda_gate == GDR_KDA_GATE_SIGMOID) memcpy(&t.v[10], &sh->gate_scale, 4);
    t.v[11] = sh->cu_seqlens != nullptr;
    t.v[12] = h0 != nullptr;
    t.v[13] = orig_dim;  // the caller's head dim (64 runs zero-padded to 128)
    return t;
}

// writes the whole header (the tag, then zeros up to GDR_STATES_HEADER_BYTES)
__global__ void k_states_tag(int* hdr, const StatesTag t) {
    for (int i = threadIdx.x; i < GDR_STATES_HEADER_BYTES / 4; i += blockDim.x) hdr[i] = i < 16 ? t.v[i] : 0;
}

// Every kernel runs on 128 channels (head_dim 64 is zero-padded to 128 by the entry
// points); the gate variant picks the prep and main kernels.
cudaError_t launch_prep(const Params& p, cudaStream_t s) {
    if (p.max_chunks == 0) return cudaSuccess;
    if (p.D != 128) return cudaErrorInvalidValue;
    return p.kda ? launch_prep_kda(p, s) : launch_prep_gdn(p, s);
}
cudaError_t launch_states(const Params& p, bool fwd, bool bwd, cudaStream_t s) {
    if (p.D != 128) return cudaErrorInvalidValue;
    return launch_states_tc(p, fwd, bwd, s);
}
cudaError_t launch_main(const Params& p, cudaStream_t s) {
    if (p.max_chunks == 0) return cudaSuccess;
    if (p.D != 128) return cudaErrorInvalidValue;
    return p.kda ? launch_main_kda(p, s) : launch_main_gdn(p, s);
}

cudaError_t launch_chunk_table(const Params& p, cudaStream_t s) {
    k_chunk_table<<<1, 1024, 0, s>>>(p.cu_seqlens, p.N, p.T_total, const_cast<int*>(p.chunk_off), p.status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
struct Layout {
    int64_t max_chunks;
    size_t status, chunk_off, W, U, Kr, R, Rlo, T, AP, gT, egT, S0, dS, segL, segLb, segP, segS, dqk, total;
    int seg_G, seg_G1;  // segments for calls that run both state directions / one
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static gdr_status check_shape(const gdr_shape* sh) {
    if (!sh) return fail(GDR_ERR_INVALID, "shape is NULL");
    if (sh->num_seqs < 1 || sh->num_heads < 1 || sh->total_tokens < 0)
        return fail(GDR_ERR_INVALID, "num_seqs and num_heads must be >= 1, total_tokens >= 0");
    if (sh->head_dim != 64 && sh->head_dim != 128)
        return fail(GDR_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (!sh->cu_seqlens && sh->total_tokens % sh->num_seqs != 0)
        return fail(GDR_ERR_INVALID, "dense layout needs total_tokens divisible by num_seqs");
    if (sh->num_heads > 65535) return fail(GDR_ERR_INVALID, "num_heads must be <= 65535");
    if (sh->num_k_heads < 0 || (sh->num_k_heads > 0 && sh->num_heads % sh->num_k_heads != 0))
        return fail(GDR_ERR_INVALID, "num_heads must be a multiple of num_k_heads (or num_k_heads 0)");
    if (sh->kda_gate != GDR_KDA_GATE_SOFTPLUS && sh->kda_gate != GDR_KDA_GATE_SIGMOID)
        return fail(GDR_ERR_INVALID, "kda_gate must be GDR_KDA_GATE_SOFTPLUS or GDR_KDA_GATE_SIGMOID");
    if (sh->kda_gate == GDR_KDA_GATE_SIGMOID && !(sh->gate_scale <= 0.f && sh->gate_scale > -1e30f))
        return fail(GDR_ERR_INVALID, "gate_scale must be finite and <= 0 (a decaying gate)");
    const int64_t N = sh->num_seqs, T = sh->total_tokens;
    const int64_t mc = sh->cu_seqlens ? (T + (CH - 1) * N) / CH : N * ((T / N + CH - 1) / CH);
    // (the kernels address per chunk-head tiles by 32-bit row: chunk-heads x 192 rows, the A / P
    // block of the KDA backward, must fit)
    if (mc > (int64_t)1 << 30 || N * sh->num_heads * (sh->head_dim / 16) > ((int64_t)1 << 31) - 1 ||
        mc * sh->num_heads * 192 > ((int64_t)1 << 31) - 1)
        return fail(GDR_ERR_INVALID, "problem too large for one call");
    return GDR_OK;
}

// Segments of the time-parallel state passing (1 = the serial chains), for calls that run
// both directions or one.  A function of the shape only, sized for one wave of about 150
// SMs: phase 1 runs 3G - 4 CTAs per (sequence, head) for both directions and 2G - 3 for
// one, phase 3 runs G - 1 per direction; each segment keeps at least 32 chunks, and G <= 8
// keeps the serial boundary composition short.
static int seg_count(const gdr_shape* sh, int64_t max_chunks, bool two_dirs) {
    if (sh->head_dim != 128) return 1;
    const int64_t pairs = (int64_t)sh->num_seqs * sh->num_heads;
    const int64_t per_seq = max_chunks / sh->num_seqs;
    int G = 1;
    for (int g = 2; g <= 8; ++g) {
        const int64_t p1 = two_dirs ? 3 * g - 4 : 2 * g - 3, p3 = two_dirs ? 2 * g - 2 : g - 1;
        if (p1 * pairs <= 148 && p3 * pairs <= 148 && per_seq >= 32 * g) G = g;
    }
    return G;
}

static Layout layout(const gdr_shape* sh) {
    Layout L{};
    const int64_t N = sh->num_seqs, H = sh->num_heads, D = sh->head_dim, T = sh->total_tokens;
    if (sh->cu_seqlens) L.max_chunks = (T + (CH - 1) * N) / CH;
    else L.max_chunks = N * ((T / N + CH - 1) / CH);
    const size_t mc = (size_t)L.max_chunks;
    size_t o = 0;
    L.status = o; o = align256(o + 16);
    L.chunk_off = o; o = align256(o + 4 * (size_t)(N + 1));
    L.W = o; o = align256(o + mc * H * CH * D * 2);
    L.U = o; o = align256(o + mc * H * CH * D * 2);
    L.Kr = o; o = align256(o + mc * H * CH * D * 2);
    L.R = o; o = align256(o + mc * H * CH * D * 2);
    L.Rlo = o; o = align256(o + mc * H * CH * D * 2);
    L.T = o; o = align256(o + mc * H * CH * CH * 2);
    L.AP = o; o = align256(o + mc * H * 3 * CH * CH * 2);  // A, P hi, P lo (the KDA backward's)
    L.gT = o; o = align256(o + mc * H * D * 4);
    L.egT = o; o = align256(o + mc * H * D * 4);
    L.S0 = o; o = align256(o + mc * H * D * D * 2);
    L.dS = o; o = align256(o + mc * H * D * D * 2);
    L.seg_G = seg_count(sh, L.max_chunks, true);
    L.seg_G1 = seg_count(sh, L.max_chunks, false);
    const int64_t Gmax = L.seg_G > L.seg_G1 ? L.seg_G : L.seg_G1;
    const size_t segb = Gmax > 1 ? (size_t)N * H * Gmax * D * D * 4 : 0;  // fp32 [pair][G][D][D]
    L.segL = o; o = align256(o + segb);
    L.segLb = o; o = align256(o + segb);
    L.segP = o; o = align256(o + segb);
    L.segS = o; o = align256(o + 2 * segb);
    // GQA: per-value-head dq, dk terms (bf16 [T, H, D] each) before the group sums
    const bool gqa = sh->num_k_heads > 0 && sh->num_k_heads < sh->num_heads;
    L.dqk = o; o = align256(o + (gqa ? 2 * (size_t)T * H * D * 2 : 0));
    L.total = o;
    return L;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

#define NEED(ptr)                                                                    \
    do {                                                                             \
        if (!(ptr)) return fail(GDR_ERR_INVALID, "required pointer %s is NULL", #ptr); \
        if (!aligned16(ptr)) return fail(GDR_ERR_INVALID, "pointer %s is not 16-byte aligned", #ptr); \
    } while (0)
#define OPT(ptr)                                                                     \
    do {                                                                             \
        if ((ptr) && !aligned16(ptr)) return fail(GDR_ERR_INVALID, "pointer %s is not 16-byte aligned", #ptr); \
    } while (0)

static void base_params(Params& p, const gdr_shape* sh, const Layout& L, void* ws, int kda) {
    memset(&p, 0, sizeof(p));
    p.N = sh->num_seqs;
    p.H = sh->num_heads;
    p.Hk = sh->num_k_heads > 0 ? sh->num_k_heads : sh->num_heads;
    p.D = sh->head_dim;
    p.T_total = sh->total_tokens;
    p.seq_len = sh->cu_seqlens ? 0 : sh->total_tokens / sh->num_seqs;
    p.max_chunks = (int)L.max_chunks;
    p.cu_seqlens = sh->cu_seqlens;
    p.scale = sh->scale;
    p.kda = kda;
    p.kda_gate = sh->kda_gate;
    p.gate_scale = sh->gate_scale;
    unsigned char* w = static_cast<unsigned char*>(ws);
    p.status = reinterpret_cast<int*>(w + L.status);
    p.chunk_off = sh->cu_seqlens ? reinterpret_cast<int*>(w + L.chunk_off) : nullptr;
    p.W = reinterpret_cast<__nv_bfloat16*>(w + L.W);
    p.U = reinterpret_cast<__nv_bfloat16*>(w + L.U);
    p.Kr = reinterpret_cast<__nv_bfloat16*>(w + L.Kr);
    p.R = reinterpret_cast<__nv_bfloat16*>(w + L.R);
    p.Rlo = reinterpret_cast<__nv_bfloat16*>(w + L.Rlo);
    p.Tm = reinterpret_cast<__nv_bfloat16*>(w + L.T);
    p.gT = reinterpret_cast<float*>(w + L.gT);
    p.egT = reinterpret_cast<float*>(w + L.egT);
    p.S0 = reinterpret_cast<__nv_bfloat16*>(w + L.S0);
    p.dS = reinterpret_cast<__nv_bfloat16*>(w + L.dS);
    p.seg_G = L.seg_G;
    p.seg_G1 = L.seg_G1;
    p.segL = reinterpret_cast<float*>(w + L.segL);
    p.segLb = reinterpret_cast<float*>(w + L.segLb);
    p.segP = reinterpret_cast<float*>(w + L.segP);
    p.segS = reinterpret_cast<float*>(w + L.segS);
}

// ---------------------------------------------------------------------------
// optional per-kernel event timing (gdr_profile_begin / gdr_profile_end)
// ---------------------------------------------------------------------------
struct Prof {
    bool on = false;
    int max_launches = 0, n = 0;
    cudaEvent_t* ev = nullptr;  // 2 per timed section
    int* kind = nullptr;
    int* kernels = nullptr;     // kernels launched in each timed section
};
static Prof g_prof;

// Launches `f` (which launches `kernels` kernels) between two recorded events when
// profiling is on.
template <class F>
static cudaError_t timed(int kind, cudaStream_t s, F&& f, int kernels = 1) {
    if (!g_prof.on || g_prof.n >= g_prof.max_launches) return f();
    const int i = g_prof.n++;
    g_prof.kind[i] = kind;
    g_prof.kernels[i] = kernels;
    cudaEventRecord(g_prof.ev[2 * i], s);
    cudaError_t e = f();
    cudaEventRecord(g_prof.ev[2 * i + 1], s);
    return e;
}

// status reset + chunk table (+ prep)
static gdr_status common_front(const Params& p, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(p.status, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
    if (p.cu_seqlens) {
        e = timed(GDR_KERNEL_CHUNK_TABLE, s, [&] { return launch_chunk_table(p, s); });
        if (e != cudaSuccess) return cuda_fail(e, "chunk table launch");
    }
    e = timed(GDR_KERNEL_PREP, s, [&] { return launch_prep(p, s); });
    if (e != cudaSuccess) return cuda_fail(e, "prep launch");
    return GDR_OK;
}

static gdr_status fwd_states_impl128(const gdr_shape* sh, const void* q, const void* k, const void* v,
                                  const float* g, const void* g_raw, const float* A_log,
                                  const float* dt_bias, const void* beta, const float* h0,
                                  void* states, size_t states_bytes, void* ws, size_t ws_bytes,
                                  void* stream, int kda, int orig_dim) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(ws); NEED(states); OPT(h0);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); } else { NEED(g); }
    const Layout L = layout(sh);
    if (ws_bytes < L.total) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    if (states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
    Params p;
    base_params(p, sh, L, ws, kda);
    p.q = (const __nv_bfloat16*)q; p.k = (const __nv_bfloat16*)k; p.v = (const __nv_bfloat16*)v;
    p.beta_logit = (const __nv_bfloat16*)beta;
    p.g = g; p.g_raw = (const __nv_bfloat16*)g_raw; p.A_log = A_log; p.dt_bias = dt_bias;
    p.h0 = h0;
    p.S0 = reinterpret_cast<__nv_bfloat16*>(static_cast<unsigned char*>(states) + GDR_STATES_HEADER_BYTES);
    cudaStream_t s = (cudaStream_t)stream;
    gdr_status st = common_front(p, s);
    if (st != GDR_OK) return st;
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, true, false, s); },
                          states_kernel_count(p, true, false));
    if (e != cudaSuccess) return cuda_fail(e, "state recurrence launch");
    k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, L.max_chunks, orig_dim));
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "states header launch");
    g_err[0] = 0;
    return GDR_OK;
}

// forward: chunk tiles (with P), the chunk-start states and final states, the output
static gdr_status fwd_impl128(const gdr_shape* sh, const void* q, const void* k, const void* v, const float* g,
                           const void* g_raw, const float* A_log, const float* dt_bias, const void* beta,
                           const float* h0, void* o, float* ht, void* states, size_t states_bytes, void* ws,
                           size_t ws_bytes, void* stream, int kda, int orig_dim) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(ws); NEED(o); OPT(h0); OPT(ht); OPT(states);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); } else { NEED(g); }
    const Layout L = layout(sh);
    if (ws_bytes < L.total) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    if (states && states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
    Params p;
    base_params(p, sh, L, ws, kda);
    p.q = (const __nv_bfloat16*)q; p.k = (const __nv_bfloat16*)k; p.v = (const __nv_bfloat16*)v;
    p.beta_logit = (const __nv_bfloat16*)beta;
    p.g = g; p.g_raw = (const __nv_bfloat16*)g_raw; p.A_log = A_log; p.dt_bias = dt_bias;
    p.h0 = h0;
    p.o = (__nv_bfloat16*)o;
    p.ht = ht;
    if (states)
        p.S0 = reinterpret_cast<__nv_bfloat16*>(static_cast<unsigned char*>(states) + GDR_STATES_HEADER_BYTES);
    p.Pm = p.dS;  // the state-gradient tiles of the backward are free in a forward call
    cudaStream_t s = (cudaStream_t)stream;
    gdr_status st = common_front(p, s);
    if (st != GDR_OK) return st;
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, true, false, s); },
                          states_kernel_count(p, true, false));
    if (e != cudaSuccess) return cuda_fail(e, "state recurrence launch");
    e = timed(GDR_KERNEL_OUT, s, [&] { return launch_out(p, s); });
    if (e != cudaSuccess) return cuda_fail(e, "output launch");
    if (states) {
        k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, L.max_chunks, orig_dim));
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "states header launch");
    }
    g_err[0] = 0;
    return GDR_OK;
}

static std::atomic<int> g_test_stall{0};  // gdr_test_stall_next_call: CTA index + 1, or 0

static gdr_status bwd_impl128(const gdr_shape* sh, const void* q, const void* k, const void* v,
                           const float* g, const void* g_raw, const float* A_log, const float* dt_bias,
                           const void* beta, const float* h0, const void* dO, const float* dht,
                           const void* states, void* ws, size_t ws_bytes, void* dq, void* dk, void* dv,
                           float* dg, void* dg_raw, void* dbeta, float* dh0, float* dA_log,
                           float* ddt_bias, void* stream, int kda, int orig_dim) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(dO); NEED(ws);
    NEED(dq); NEED(dk); NEED(dv); NEED(dbeta); NEED(dh0);
    OPT(h0); OPT(dht); OPT(states);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); NEED(dg_raw); NEED(dA_log); NEED(ddt_bias); }
    else { NEED(g); NEED(dg); }
    const Layout L = layout(sh);
    if (ws_bytes < L.total) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    Params p;
    base_params(p, sh, L, ws, kda);
    p.q = (const __nv_bfloat16*)q; p.k = (const __nv_bfloat16*)k; p.v = (const __nv_bfloat16*)v;
    p.dO = (const __nv_bfloat16*)dO; p.beta_logit = (const __nv_bfloat16*)beta;
    p.g = g; p.g_raw = (const __nv_bfloat16*)g_raw; p.A_log = A_log; p.dt_bias = dt_bias;
    p.h0 = h0; p.dht = dht;
    if (states) {
        p.S0 = reinterpret_cast<__nv_bfloat16*>(const_cast<unsigned char*>(static_cast<const unsigned char*>(states)) +
                                                GDR_STATES_HEADER_BYTES);
        p.states_hdr = static_cast<const int*>(states);
        const StatesTag t = states_tag(sh, kda, h0, L.max_chunks, orig_dim);
        memcpy(p.states_tag, t.v, sizeof(t.v));
    }
    if (!kda && p.D == 128) p.test_stall = g_test_stall.exchange(0);
    p.dq = (__nv_bfloat16*)dq; p.dk = (__nv_bfloat16*)dk; p.dv = (__nv_bfloat16*)dv;
    if (p.Hk < p.H) {  // GQA: per-value-head terms in the workspace, summed over each group at the end
        p.dq_out = p.dq;
        p.dk_out = p.dk;
        p.dq = reinterpret_cast<__nv_bfloat16*>(static_cast<unsigned char*>(ws) + L.dqk);
        p.dk = p.dq + (size_t)p.T_total * p.H * p.D;
    }
    p.dbeta = (__nv_bfloat16*)dbeta; p.dg = dg; p.dg_raw = (__nv_bfloat16*)dg_raw;
    p.dh0 = dh0; p.dA_log = dA_log; p.ddt_bias = ddt_bias;
    if (kda) p.APm = reinterpret_cast<__nv_bfloat16*>(static_cast<unsigned char*>(ws) + L.AP);
    cudaStream_t s = (cudaStream_t)stream;
    if (kda) {
        cudaError_t e = cudaMemsetAsync(dA_log, 0, sizeof(float) * p.H, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * p.H * p.D, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dA_log/ddt_bias)");
    }
    gdr_status st = common_front(p, s);
    if (st != GDR_OK) return st;
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, states == nullptr, true, s); },
                          states_kernel_count(p, states == nullptr, true));
    if (e != cudaSuccess) return cuda_fail(e, "state recurrence launch");
    e = timed(GDR_KERNEL_MAIN, s, [&] { return launch_main(p, s); });
    if (e != cudaSuccess) return cuda_fail(e, "main backward launch");
    if (p.Hk < p.H) {
        e = timed(GDR_KERNEL_MAIN, s, [&] { return launch_group_sum(p, s); });
        if (e != cudaSuccess) return cuda_fail(e, "group sum launch");
    }
    g_err[0] = 0;
    return GDR_OK;
}

// ---------------------------------------------------------------------------
// head_dim 64: the same tcgen05 kernels on channels zero-padded to 128
//
// A zero key channel adds nothing to any product and keeps its row of the state at zero
// from a zero start (k has no component there, so the delta update never writes it), and
// a zero value channel keeps its column at zero; the L2 norms, dot products and channel
// sums of the method are unchanged by zero channels.  So the D = 64 problem is the
// D = 128 problem on inputs padded with zeros, and its results are the first 64 channels
// of the padded results (the padded channels' gradients are exactly zero).  The pads
// live in the workspace after the D = 128 layout; saved states keep the padded layout.
// ---------------------------------------------------------------------------

// dst[b][r][v] = src[b][r][v] for r < rin, v < vin, else 0 (pad); or the first rin rows and
// vin units of every block of src into a dense dst (unpad).  Units are 16 bytes.
__global__ void __launch_bounds__(256) k_pad16(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t nb,
                                               int rin, int vin, int rout, int vout, int unpad) {
    const int64_t per = unpad ? (int64_t)rin * vin : (int64_t)rout * vout;
    const int64_t n = nb * per;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / per;
        const int rem = (int)(i % per);
        if (unpad) {
            const int r = rem / vin, v = rem % vin;
            dst[i] = src[(b * rout + r) * vout + v];
        } else {
            const int r = rem / vout, v = rem % vout;
            dst[i] = (r < rin && v < vin) ? src[(b * rin + r) * vin + v] : make_uint4(0, 0, 0, 0);
        }
    }
}

// nb blocks of rin x cin elements of esz bytes <-> blocks of rout x cout (cin, cout: 16-byte multiples)
static cudaError_t pad_copy(const void* src, void* dst, int64_t nb, int rin, int cin, int rout, int cout, int esz,
                            bool unpad, cudaStream_t s) {
    const int64_t units = nb * (unpad ? (int64_t)rin * cin : (int64_t)rout * cout) * esz / 16;
    if (units == 0) return cudaSuccess;
    const int64_t want = (units + 255) / 256;
    const int grid = (int)(want < 8 * num_sms() ? want : 8 * num_sms());
    k_pad16<<<grid, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), nb, rin, cin * esz / 16,
                                 rout, cout * esz / 16, unpad ? 1 : 0);
    return cudaGetLastError();
}

struct Pad64 {  // byte offsets of the padded tensors, from the end of the D = 128 layout
    size_t q, k, v, dO, gr, dtb, h0, dht, dq, dk, dv, dgr, dh0, ddt, o, ht, total;
};
static gdr_shape shape128(const gdr_shape* sh) {
    gdr_shape t = *sh;
    t.head_dim = 128;
    return t;
}
static Pad64 pad64_layout(const gdr_shape* sh) {
    Pad64 P{};
    const size_t T = (size_t)sh->total_tokens, H = (size_t)sh->num_heads, N = (size_t)sh->num_seqs;
    const size_t Hk = sh->num_k_heads > 0 ? (size_t)sh->num_k_heads : H;
    const size_t tok_k = T * Hk * 128 * 2, tok = T * H * 128 * 2, st = N * H * 128 * 128 * 4, hd = H * 128 * 4;
    size_t o = 0;
    auto put = [&](size_t& f, size_t bytes) { f = o; o = align256(o + bytes); };
    put(P.q, tok_k); put(P.k, tok_k); put(P.v, tok); put(P.dO, tok); put(P.gr, tok); put(P.dtb, hd);
    put(P.h0, st); put(P.dht, st); put(P.dq, tok_k); put(P.dk, tok_k); put(P.dv, tok); put(P.dgr, tok);
    put(P.dh0, st); put(P.ddt, hd); put(P.o, tok); put(P.ht, st);
    P.total = o;
    return P;
}
// the whole workspace of a call: the layout of the kernels' shape, then (D = 64) the pads
static size_t workspace_total(const gdr_shape* sh) {
    if (sh->head_dim == 128) return layout(sh).total;
    const gdr_shape s128 = shape128(sh);
    return align256(layout(&s128).total) + pad64_layout(sh).total;
}

// The padded inputs of a D = 64 call: q, k, v (and dO, the KDA gate inputs, h0, dht when
// given) into the pad region.  `base` is the pad region; `P` its layout.
struct Pad64In {
    const void *q, *k, *v, *dO, *g_raw;
    const float *dt_bias, *h0, *dht;
};
static gdr_status pad64_inputs(const gdr_shape* sh, const Pad64& P, unsigned char* base, Pad64In& in, int kda,
                               cudaStream_t s) {
    const int64_t T = sh->total_tokens, H = sh->num_heads, N = sh->num_seqs;
    const int64_t Hk = sh->num_k_heads > 0 ? sh->num_k_heads : H;
    cudaError_t e = cudaSuccess;
    auto tok = [&](const void*& x, size_t off, int64_t heads) {
        if (!x || e != cudaSuccess) return;
        e = pad_copy(x, base + off, T * heads, 1, 64, 1, 128, 2, false, s);
        x = base + off;
    };
    tok(in.q, P.q, Hk);
    tok(in.k, P.k, Hk);
    tok(in.v, P.v, H);
    tok(in.dO, P.dO, H);
    if (kda) tok(in.g_raw, P.gr, H);
    auto st = [&](const float*& x, size_t off) {
        if (!x || e != cudaSuccess) return;
        e = pad_copy(x, base + off, N * H, 64, 64, 128, 128, 4, false, s);
        x = reinterpret_cast<const float*>(base + off);
    };
    st(in.h0, P.h0);
    st(in.dht, P.dht);
    if (kda && in.dt_bias && e == cudaSuccess) {
        e = pad_copy(in.dt_bias, base + P.dtb, H, 1, 64, 1, 128, 4, false, s);
        in.dt_bias = reinterpret_cast<const float*>(base + P.dtb);
    }
    return e == cudaSuccess ? GDR_OK : cuda_fail(e, "channel padding launch");
}

// Calls with no token at all (every sequence empty): nothing to differentiate but h0, whose
// gradient is dht; the final state of a forward is h0.  The token tensors may be NULL.
static gdr_status empty_state_copy(float* dst, const float* src, const gdr_shape* sh, cudaStream_t s) {
    const size_t bytes = (size_t)sh->num_seqs * sh->num_heads * sh->head_dim * sh->head_dim * 4;
    cudaError_t e = src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dst, 0, bytes, s);
    return e == cudaSuccess ? GDR_OK : cuda_fail(e, "state copy (no tokens)");
}
static gdr_status empty_front(void* ws, size_t ws_bytes, const gdr_shape* sh, cudaStream_t s) {
    if (!ws) return fail(GDR_ERR_INVALID, "required pointer ws is NULL%s");
    if (ws_bytes < workspace_total(sh)) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int), s);
    return e == cudaSuccess ? GDR_OK : cuda_fail(e, "cudaMemsetAsync(status)");
}

static gdr_status fwd_states_impl(const gdr_shape* sh, const void* q, const void* k, const void* v,
                                  const float* g, const void* g_raw, const float* A_log,
                                  const float* dt_bias, const void* beta, const float* h0,
                                  void* states, size_t states_bytes, void* ws, size_t ws_bytes,
                                  void* stream, int kda) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    if (sh->total_tokens == 0) {
        NEED(states); OPT(h0);
        if (states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
        cudaStream_t s = (cudaStream_t)stream;
        if (gdr_status st = empty_front(ws, ws_bytes, sh, s)) return st;
        k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, 0, sh->head_dim));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "states header launch");
        g_err[0] = 0;
        return GDR_OK;
    }
    if (sh->head_dim == 128)
        return fwd_states_impl128(sh, q, k, v, g, g_raw, A_log, dt_bias, beta, h0, states, states_bytes, ws,
                                  ws_bytes, stream, kda, 128);
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(ws); NEED(states); OPT(h0);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); } else { NEED(g); }
    const gdr_shape s128 = shape128(sh);
    if (gdr_status st1 = check_shape(&s128)) return st1;
    if (ws_bytes < workspace_total(sh)) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    if (states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
    const size_t inner = align256(layout(&s128).total);
    unsigned char* base = static_cast<unsigned char*>(ws) + inner;
    Pad64In in{q, k, v, nullptr, g_raw, dt_bias, h0, nullptr};
    cudaStream_t s = (cudaStream_t)stream;
    if (gdr_status st = pad64_inputs(sh, pad64_layout(sh), base, in, kda, s)) return st;
    return fwd_states_impl128(&s128, in.q, in.k, in.v, g, in.g_raw, A_log, in.dt_bias, beta, in.h0, states,
                              states_bytes, ws, inner, stream, kda, 64);
}

static gdr_status fwd_impl(const gdr_shape* sh, const void* q, const void* k, const void* v, const float* g,
                           const void* g_raw, const float* A_log, const float* dt_bias, const void* beta,
                           const float* h0, void* o, float* ht, void* states, size_t states_bytes, void* ws,
                           size_t ws_bytes, void* stream, int kda) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    if (sh->total_tokens == 0) {
        OPT(h0); OPT(ht); OPT(states);
        if (states && states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
        cudaStream_t s = (cudaStream_t)stream;
        if (gdr_status st = empty_front(ws, ws_bytes, sh, s)) return st;
        if (ht)
            if (gdr_status st = empty_state_copy(ht, h0, sh, s)) return st;
        if (states) {
            k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, 0, sh->head_dim));
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return cuda_fail(e, "states header launch");
        }
        g_err[0] = 0;
        return GDR_OK;
    }
    if (sh->head_dim == 128)
        return fwd_impl128(sh, q, k, v, g, g_raw, A_log, dt_bias, beta, h0, o, ht, states, states_bytes, ws, ws_bytes,
                           stream, kda, 128);
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(ws); NEED(o); OPT(h0); OPT(ht); OPT(states);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); } else { NEED(g); }
    const gdr_shape s128 = shape128(sh);
    if (gdr_status st1 = check_shape(&s128)) return st1;
    if (ws_bytes < workspace_total(sh)) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    if (states && states_bytes < gdr_states_bytes(sh)) return fail(GDR_ERR_WORKSPACE, "states buffer too small%s");
    const size_t inner = align256(layout(&s128).total);
    unsigned char* base = static_cast<unsigned char*>(ws) + inner;
    const Pad64 P = pad64_layout(sh);
    Pad64In in{q, k, v, nullptr, g_raw, dt_bias, h0, nullptr};
    cudaStream_t s = (cudaStream_t)stream;
    if (gdr_status st = pad64_inputs(sh, P, base, in, kda, s)) return st;
    float* htp = ht ? reinterpret_cast<float*>(base + P.ht) : nullptr;
    gdr_status st = fwd_impl128(&s128, in.q, in.k, in.v, g, in.g_raw, A_log, in.dt_bias, beta, in.h0, base + P.o, htp,
                                states, states_bytes, ws, inner, stream, kda, 64);
    if (st != GDR_OK) return st;
    const int64_t T = sh->total_tokens, H = sh->num_heads, N = sh->num_seqs;
    cudaError_t e = pad_copy(base + P.o, o, T * H, 1, 64, 1, 128, 2, true, s);
    if (e == cudaSuccess && ht) e = pad_copy(htp, ht, N * H, 64, 64, 128, 128, 4, true, s);
    return e == cudaSuccess ? GDR_OK : cuda_fail(e, "channel unpadding launch");
}

static gdr_status bwd_impl(const gdr_shape* sh, const void* q, const void* k, const void* v,
                           const float* g, const void* g_raw, const float* A_log, const float* dt_bias,
                           const void* beta, const float* h0, const void* dO, const float* dht,
                           const void* states, void* ws, size_t ws_bytes, void* dq, void* dk, void* dv,
                           float* dg, void* dg_raw, void* dbeta, float* dh0, float* dA_log,
                           float* ddt_bias, void* stream, int kda) {
    if (gdr_status st0 = check_shape(sh)) return st0;
    if (sh->total_tokens == 0) {
        NEED(dh0); OPT(h0); OPT(dht); OPT(states);
        if (kda) { NEED(A_log); NEED(dt_bias); NEED(dA_log); NEED(ddt_bias); }
        cudaStream_t s = (cudaStream_t)stream;
        if (gdr_status st = empty_front(ws, ws_bytes, sh, s)) return st;
        if (gdr_status st = empty_state_copy(dh0, dht, sh, s)) return st;
        if (kda) {
            cudaError_t e = cudaMemsetAsync(dA_log, 0, sizeof(float) * sh->num_heads, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * sh->num_heads * sh->head_dim, s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dA_log/ddt_bias)");
        }
        g_err[0] = 0;
        return GDR_OK;
    }
    if (sh->head_dim == 128)
        return bwd_impl128(sh, q, k, v, g, g_raw, A_log, dt_bias, beta, h0, dO, dht, states, ws, ws_bytes, dq, dk, dv,
                           dg, dg_raw, dbeta, dh0, dA_log, ddt_bias, stream, kda, 128);
    NEED(q); NEED(k); NEED(v); NEED(beta); NEED(dO); NEED(ws);
    NEED(dq); NEED(dk); NEED(dv); NEED(dbeta); NEED(dh0);
    OPT(h0); OPT(dht); OPT(states);
    if (kda) { NEED(g_raw); NEED(A_log); NEED(dt_bias); NEED(dg_raw); NEED(dA_log); NEED(ddt_bias); }
    else { NEED(g); NEED(dg); }
    const gdr_shape s128 = shape128(sh);
    if (gdr_status st1 = check_shape(&s128)) return st1;
    if (ws_bytes < workspace_total(sh)) return fail(GDR_ERR_WORKSPACE, "workspace too small%s");
    const size_t inner = align256(layout(&s128).total);
    unsigned char* base = static_cast<unsigned char*>(ws) + inner;
    const Pad64 P = pad64_layout(sh);
    Pad64In in{q, k, v, dO, g_raw, dt_bias, h0, dht};
    cudaStream_t s = (cudaStream_t)stream;
    if (gdr_status st = pad64_inputs(sh, P, base, in, kda, s)) return st;
    gdr_status st = bwd_impl128(&s128, in.q, in.k, in.v, g, in.g_raw, A_log, in.dt_bias, beta, in.h0, in.dO, in.dht,
                                states, ws, inner, base + P.dq, base + P.dk, base + P.dv, dg,
                                kda ? base + P.dgr : nullptr, dbeta, reinterpret_cast<float*>(base + P.dh0), dA_log,
                                kda ? reinterpret_cast<float*>(base + P.ddt) : nullptr, stream, kda, 64);
    if (st != GDR_OK) return st;
    const int64_t T = sh->total_tokens, H = sh->num_heads, N = sh->num_seqs;
    const int64_t Hk = sh->num_k_heads > 0 ? sh->num_k_heads : H;
    cudaError_t e = pad_copy(base + P.dq, dq, T * Hk, 1, 64, 1, 128, 2, true, s);
    if (e == cudaSuccess) e = pad_copy(base + P.dk, dk, T * Hk, 1, 64, 1, 128, 2, true, s);
    if (e == cudaSuccess) e = pad_copy(base + P.dv, dv, T * H, 1, 64, 1, 128, 2, true, s);
    if (e == cudaSuccess) e = pad_copy(base + P.dh0, dh0, N * H, 64, 64, 128, 128, 4, true, s);
    if (kda && e == cudaSuccess) e = pad_copy(base + P.dgr, dg_raw, T * H, 1, 64, 1, 128, 2, true, s);
    if (kda && e == cudaSuccess) e = pad_copy(base + P.ddt, ddt_bias, H, 1, 64, 1, 128, 4, true, s);
    return e == cudaSuccess ? GDR_OK : cuda_fail(e, "channel unpadding launch");
}

}  // namespace gdr

using namespace gdr;

extern "C" {

size_t gdr_workspace_bytes(const gdr_shape* shape) {
    if (check_shape(shape) != GDR_OK) return 0;
    return workspace_total(shape);
}

size_t gdr_states_bytes(const gdr_shape* shape) {
    if (check_shape(shape) != GDR_OK) return 0;
    const Layout L = layout(shape);
    // (head_dim 64 keeps its states in the layout of the zero-padded 128-channel problem)
    return GDR_STATES_HEADER_BYTES + (size_t)L.max_chunks * shape->num_heads * 128 * 128 * 2;
}

void gdr_test_stall_next_call(int cta) { g_test_stall.store(cta >= 0 ? cta + 1 : 0); }

gdr_status gdr_fwd_states(const gdr_shape* shape, const void* q, const void* k, const void* v,
                          const float* g, const void* beta_logit, const float* h0, void* states,
                          size_t states_bytes, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_states_impl(shape, q, k, v, g, nullptr, nullptr, nullptr, beta_logit, h0, states,
                           states_bytes, workspace, workspace_bytes, stream, 0);
}

gdr_status kda_fwd_states(const gdr_shape* shape, const void* q, const void* k, const void* v,
                          const void* g_raw, const float* A_log, const float* dt_bias,
                          const void* beta_logit, const float* h0, void* states, size_t states_bytes,
                          void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_states_impl(shape, q, k, v, nullptr, g_raw, A_log, dt_bias, beta_logit, h0, states,
                           states_bytes, workspace, workspace_bytes, stream, 1);
}

gdr_status gdr_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v, const float* g,
                   const void* beta_logit, const float* h0, void* o, float* ht, void* states,
                   size_t states_bytes, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(shape, q, k, v, g, nullptr, nullptr, nullptr, beta_logit, h0, o, ht, states, states_bytes,
                    workspace, workspace_bytes, stream, 0);
}

gdr_status kda_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v, const void* g_raw,
                   const float* A_log, const float* dt_bias, const void* beta_logit, const float* h0, void* o,
                   float* ht, void* states, size_t states_bytes, void* workspace, size_t workspace_bytes,
                   void* stream) {
    return fwd_impl(shape, q, k, v, nullptr, g_raw, A_log, dt_bias, beta_logit, h0, o, ht, states, states_bytes,
                    workspace, workspace_bytes, stream, 1);
}

gdr_status gdr_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v, const float* g,
                   const void* beta_logit, const float* h0, const void* dO, const float* dht,
                   const void* states, void* workspace, size_t workspace_bytes, void* dq, void* dk,
                   void* dv, float* dg, void* dbeta, float* dh0, void* stream) {
    return bwd_impl(shape, q, k, v, g, nullptr, nullptr, nullptr, beta_logit, h0, dO, dht, states,
                    workspace, workspace_bytes, dq, dk, dv, dg, nullptr, dbeta, dh0, nullptr, nullptr,
                    stream, 0);
}

gdr_status kda_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v, const void* g_raw,
                   const float* A_log, const float* dt_bias, const void* beta_logit, const float* h0,
                   const void* dO, const float* dht, const void* states, void* workspace,
                   size_t workspace_bytes, void* dq, void* dk, void* dv, void* dg_raw, void* dbeta,
                   float* dh0, float* dA_log, float* ddt_bias, void* stream) {
    return bwd_impl(shape, q, k, v, nullptr, g_raw, A_log, dt_bias, beta_logit, h0, dO, dht, states,
                    workspace, workspace_bytes, dq, dk, dv, nullptr, dg_raw, dbeta, dh0, dA_log, ddt_bias,
                    stream, 1);
}

gdr_status gdr_conv1d_bwd(int32_t num_seqs, int64_t total_tokens, int32_t channels, int32_t width,
                          const int64_t* cu_seqlens, const void* x, const float* weight, const float* bias,
                          const void* dy, int32_t silu, void* dx, float* dweight, float* dbias, void* stream) {
    if (num_seqs < 1 || total_tokens < 0 || channels < 1)
        return fail(GDR_ERR_INVALID, "num_seqs and channels must be >= 1, total_tokens >= 0%s");
    if (width < 1 || width > 4) return fail(GDR_ERR_UNSUPPORTED, "width must be 1 to 4%s");
    if (channels % 2 != 0) return fail(GDR_ERR_INVALID, "channels must be even%s");
    if (!cu_seqlens && total_tokens % num_seqs != 0)
        return fail(GDR_ERR_INVALID, "dense layout needs total_tokens divisible by num_seqs%s");
    if ((int64_t)channels * total_tokens > ((int64_t)1 << 40)) return fail(GDR_ERR_INVALID, "problem too large%s");
    NEED(x); NEED(weight); NEED(dy); NEED(dx); NEED(dweight); OPT(bias); OPT(dbias);
    ConvParams p;
    p.N = num_seqs;
    p.T = total_tokens;
    p.C = channels;
    p.K = width;
    p.silu = silu != 0;
    p.cu_seqlens = cu_seqlens;
    p.x = (const __nv_bfloat16*)x;
    p.dy = (const __nv_bfloat16*)dy;
    p.w = weight;
    p.bias = bias;
    p.dx = (__nv_bfloat16*)dx;
    p.dw = dweight;
    p.dbias = dbias;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(dweight, 0, sizeof(float) * channels * width, s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, sizeof(float) * channels, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dweight/dbias)");
    e = timed(GDR_KERNEL_CONV, s, [&] { return launch_conv1d_bwd(p, s); });
    if (e != cudaSuccess) return cuda_fail(e, "conv1d backward launch");
    g_err[0] = 0;
    return GDR_OK;
}

gdr_status gdr_workspace_status(const void* workspace, void* stream, int* device_status) {
    if (!workspace || !device_status) return fail(GDR_ERR_INVALID, "workspace and device_status must be non-NULL%s");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
    *device_status = v;
    return GDR_OK;
}

const char* gdr_last_error(void) { return g_err; }

gdr_status gdr_profile_begin(int max_launches) {
    if (max_launches <= 0) return fail(GDR_ERR_INVALID, "max_launches must be > 0%s");
    if (g_prof.ev) {
        for (int i = 0; i < 2 * g_prof.max_launches; ++i) cudaEventDestroy(g_prof.ev[i]);
        delete[] g_prof.ev;
        delete[] g_prof.kind;
        delete[] g_prof.kernels;
    }
    g_prof = Prof();
    g_prof.ev = new cudaEvent_t[2 * max_launches];
    g_prof.kind = new int[max_launches];
    g_prof.kernels = new int[max_launches];
    for (int i = 0; i < 2 * max_launches; ++i) {
        cudaError_t e = cudaEventCreate(&g_prof.ev[i]);
        if (e != cudaSuccess) {
            g_prof.max_launches = i / 2;
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    g_prof.max_launches = max_launches;
    g_prof.on = true;
    return GDR_OK;
}

gdr_status gdr_profile_end(double* total_ms, int* launches) {
    if (!total_ms || !launches) return fail(GDR_ERR_INVALID, "output arrays must be non-NULL%s");
    for (int k = 0; k < GDR_KERNEL_COUNT; ++k) { total_ms[k] = 0.0; launches[k] = 0; }
    g_prof.on = false;
    for (int i = 0; i < g_prof.n; ++i) {
        cudaError_t e = cudaEventSynchronize(g_prof.ev[2 * i + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
        float ms = 0.f;
        e = cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
        total_ms[g_prof.kind[i]] += ms;
        launches[g_prof.kind[i]] += g_prof.kernels[i];
    }
    g_prof.n = 0;
    return GDR_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gdr_bwd_fixed: the GDN backward with its scratch in a static device array.
//
// Some callers cannot allocate device memory where they run the backward: a
// plug-in whose host framework owns every device allocation and hands the
// plug-in only tensors, or code on a path where a cudaMalloc (which may
// synchronise the device or fail under memory pressure) is not allowed.  For
// them this entry point needs no workspace argument: its scratch is the array
// below, which every GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_fixed_ws[GDR_FIXED_WORKSPACE_BYTES];

namespace gdr {
static std::mutex g_fixed_mu;
static void* g_fixed_addr[GDR_FIXED_MAX_DEVICES];

// Device address of g_fixed_ws on the current device (resolved once per device).
static gdr_status fixed_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= GDR_FIXED_MAX_DEVICES) return fail(GDR_ERR_UNSUPPORTED, "device index out of range%s");
    std::lock_guard<std::mutex> lock(g_fixed_mu);
    if (!g_fixed_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fixed_ws);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(fixed workspace)");
        g_fixed_addr[dev] = p;
    }
    *out = g_fixed_addr[dev];
    return GDR_OK;
}
}  // namespace gdr

extern "C" gdr_status gdr_bwd_fixed(const gdr_shape* shape, const void* q, const void* k, const void* v,
                                    const float* g, const void* beta_logit, const float* h0, const void* dO,
                                    const float* dht, const void* states, void* dq, void* dk, void* dv,
                                    float* dg, void* dbeta, float* dh0, void* stream) {
    if (gdr_status st0 = check_shape(shape)) return st0;
    const size_t need = workspace_total(shape);
    if (need > (size_t)GDR_FIXED_WORKSPACE_BYTES) {
        snprintf(g_err, sizeof(g_err),
                 "gdr_bwd_fixed: this problem needs %zu bytes of scratch; the fixed workspace holds %zu "
                 "(use gdr_bwd with a caller workspace)",
                 need, (size_t)GDR_FIXED_WORKSPACE_BYTES);
        return GDR_ERR_WORKSPACE;
    }
    void* ws = nullptr;
    if (gdr_status st1 = fixed_workspace(&ws)) return st1;
    // The status word is the only scratch that must start at zero; bwd_impl
    // clears it on the stream before any kernel runs.  Everything else in the
    // scratch is fully written before it is read within one call.
    return bwd_impl(shape, q, k, v, g, nullptr, nullptr, nullptr, beta_logit, h0, dO, dht, states, ws,
                    (size_t)GDR_FIXED_WORKSPACE_BYTES, dq, dk, dv, dg, nullptr, dbeta, dh0, nullptr, nullptr,
                    stream, 0);
}
