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
static StatesTag states_tag(const gdr_shape* sh, int kda, const float* h0, int64_t max_chunks) {
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
    return t;
}

// writes the whole header (the tag, then zeros up to GDR_STATES_HEADER_BYTES)
__global__ void k_states_tag(int* hdr, const StatesTag t) {
    for (int i = threadIdx.x; i < GDR_STATES_HEADER_BYTES / 4; i += blockDim.x) hdr[i] = i < 16 ? t.v[i] : 0;
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
    size_t status, chunk_off, W, U, Kr, R, Rlo, T, gT, egT, S0, dS, segL, segLb, segP, segS, dqk, total;
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
    // (the kernels address per chunk-head tiles by 32-bit row: chunk-heads x 128 rows must fit)
    if (mc > (int64_t)1 << 30 || N * sh->num_heads * (sh->head_dim / 16) > ((int64_t)1 << 31) - 1 ||
        mc * sh->num_heads * 128 > ((int64_t)1 << 31) - 1)
        return fail(GDR_ERR_INVALID, "problem too large for one call");
    return GDR_OK;
}

// Segments of the time-parallel state passing (1 = the serial chains), for calls that run
// both directions or one.  A function of the shape only, sized for one wave of about 150
// SMs: phase 1 runs 3G - 4 CTAs per (sequence, head) for both directions and 2G - 3 for
// one, phase 3 runs G per direction; each segment keeps at least 32 chunks, and G <= 8
// keeps the serial boundary composition short.
static int seg_count(const gdr_shape* sh, int64_t max_chunks, bool two_dirs) {
    if (sh->head_dim != 128) return 1;
    const int64_t pairs = (int64_t)sh->num_seqs * sh->num_heads;
    const int64_t per_seq = max_chunks / sh->num_seqs;
    int G = 1;
    for (int g = 2; g <= 8; ++g) {
        const int64_t p1 = two_dirs ? 3 * g - 4 : 2 * g - 3, p3 = two_dirs ? 2 * g : g;
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
    cudaEvent_t* ev = nullptr;  // 2 per launch
    int* kind = nullptr;
};
static Prof g_prof;

// Launches `f` between two recorded events when profiling is on.
template <class F>
static cudaError_t timed(int kind, cudaStream_t s, F&& f) {
    if (!g_prof.on || g_prof.n >= g_prof.max_launches) return f();
    const int i = g_prof.n++;
    g_prof.kind[i] = kind;
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

static gdr_status fwd_states_impl(const gdr_shape* sh, const void* q, const void* k, const void* v,
                                  const float* g, const void* g_raw, const float* A_log,
                                  const float* dt_bias, const void* beta, const float* h0,
                                  void* states, size_t states_bytes, void* ws, size_t ws_bytes,
                                  void* stream, int kda) {
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
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, true, false, s); });
    if (e != cudaSuccess) return cuda_fail(e, "state recurrence launch");
    k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, L.max_chunks));
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "states header launch");
    g_err[0] = 0;
    return GDR_OK;
}

// forward: chunk tiles (with P), the chunk-start states and final states, the output
static gdr_status fwd_impl(const gdr_shape* sh, const void* q, const void* k, const void* v, const float* g,
                           const void* g_raw, const float* A_log, const float* dt_bias, const void* beta,
                           const float* h0, void* o, float* ht, void* states, size_t states_bytes, void* ws,
                           size_t ws_bytes, void* stream, int kda) {
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
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, true, false, s); });
    if (e != cudaSuccess) return cuda_fail(e, "state recurrence launch");
    e = timed(GDR_KERNEL_OUT, s, [&] { return launch_out(p, s); });
    if (e != cudaSuccess) return cuda_fail(e, "output launch");
    if (states) {
        k_states_tag<<<1, 32, 0, s>>>(static_cast<int*>(states), states_tag(sh, kda, h0, L.max_chunks));
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "states header launch");
    }
    g_err[0] = 0;
    return GDR_OK;
}

static std::atomic<int> g_test_stall{0};  // gdr_test_stall_next_call: CTA index + 1, or 0

static gdr_status bwd_impl(const gdr_shape* sh, const void* q, const void* k, const void* v,
                           const float* g, const void* g_raw, const float* A_log, const float* dt_bias,
                           const void* beta, const float* h0, const void* dO, const float* dht,
                           const void* states, void* ws, size_t ws_bytes, void* dq, void* dk, void* dv,
                           float* dg, void* dg_raw, void* dbeta, float* dh0, float* dA_log,
                           float* ddt_bias, void* stream, int kda) {
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
        const StatesTag t = states_tag(sh, kda, h0, L.max_chunks);
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
    cudaStream_t s = (cudaStream_t)stream;
    if (kda) {
        cudaError_t e = cudaMemsetAsync(dA_log, 0, sizeof(float) * p.H, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * p.H * p.D, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(dA_log/ddt_bias)");
    }
    gdr_status st = common_front(p, s);
    if (st != GDR_OK) return st;
    cudaError_t e = timed(GDR_KERNEL_STATES, s, [&] { return launch_states(p, states == nullptr, true, s); });
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

}  // namespace gdr

using namespace gdr;

extern "C" {

size_t gdr_workspace_bytes(const gdr_shape* shape) {
    if (check_shape(shape) != GDR_OK) return 0;
    return layout(shape).total;
}

size_t gdr_states_bytes(const gdr_shape* shape) {
    if (check_shape(shape) != GDR_OK) return 0;
    const Layout L = layout(shape);
    return GDR_STATES_HEADER_BYTES + (size_t)L.max_chunks * shape->num_heads * shape->head_dim * shape->head_dim * 2;
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
    }
    g_prof = Prof();
    g_prof.ev = new cudaEvent_t[2 * max_launches];
    g_prof.kind = new int[max_launches];
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
        launches[g_prof.kind[i]] += 1;
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
    const size_t need = layout(shape).total;
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
