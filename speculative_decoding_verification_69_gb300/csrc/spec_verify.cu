// spec_verify.cu -- sm_103a kernels and C ABI of the verification step.
//
// One call of spec_verify enqueues five kernels on the caller's stream:
//   1. sv_prep    per request: clamp the verify length, validate draft tokens,
//                 decide greedy / sampled, temperature scale; list the logit
//                 rows the step must read (target 0..L, draft 0..L-1 when
//                 sampled) -- all drafts are scored from one target pass and
//                 checked together ("speculative decoding от черновика до
//                 проверки" (braintools.ru), "Как это работает", steps 2-3).
//   2. sv_pass1   the logit stream: every needed row is read once, 8 KiB per
//                 warp item through a per-warp ring of bulk copies into shared
//                 memory; per item the exact max and either the lowest-index
//                 argmax (greedy) or the sum of 2^((z - m) log2(e)/T).
//   3. sv_decide  per request: row statistics from the item partials, Philox
//                 uniforms, the acceptance rule of "Спекулятивный декодинг в
//                 проде" (kiosknews.app), "Немного теории", "Правило проверки"
//                 (argmax comparison at temperature 0), first rejection by warp
//                 ballot, accepted prefix and greedy token written.
//   4. sv_sample  per (request, 4 KiB chunk) of the one row (pair) to draw from:
//                 residual masses of max(0, p - q) (after a rejection) or of p
//                 (bonus), with exact normalisers.
//   5. sv_find    per request: inverse CDF over chunks, then over the chosen
//                 chunk's elements.
// spec_verify_early_exit runs kernels 1-3 once per wave of positions, then 4-5.
// spec_verify_tree_greedy, spec_verify_tree, spec_draft_confidence,
// spec_schedule_len and spec_schedule_budget reuse the statistics pass or are
// small kernels of their own (sv_tree_rows / sv_tree_decide, sv_tree_rows_s /
// sv_tree_walk, sv_conf_rows / sv_conf_out, sv_schedule, sv_schedule_budget).
// sv_tree_walk runs a cluster of CTAs per request: sibling candidates are
// checked against residuals kept in closed form (a threshold on
// max(0, a - s b)), one pass over the vocabulary per rejection.
#include "spec_verify.h"
#include "sv_common.cuh"
#include "lm_gemm.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

namespace sv {

constexpr double kLog2E = 1.4426950408889634074;
constexpr float kLog2EHi = 0x1.715476p+0f;   // log2(e) rounded to float
constexpr float kLog2ELo = 0x1.4ae0c0p-26f;  // log2(e) - kLog2EHi (to ~1e-16)
constexpr float kLn2F = 0.693147182f;

struct ReqInfo {
    int L;        // effective verify length
    int greedy;   // 1: temperature 0 path
    float c;      // log2(e)/T as a float (statistics pass)
    float c_hi;   // two-float log2(e)/T, c_hi rounded toward zero (sampler, acceptance)
    float c_lo;   // >= FLT_MIN
    float T;      // temperature as given
    int ord;      // sampled: the request's entry in samp_list (request order); greedy: -1
};

struct SampInfo {
    int mode;    // 1 residual at row a, 2 bonus at row L
    int slot_t;  // target row slot to sample from
    int slot_d;  // draft row slot (mode 1)
    int a;       // emitted position
    float m_t;   // max logit of the target row
    float m_d;   // max logit of the draft row (mode 1)
    float l_t;   // log2(1/S) of the target row (mode 1; 0 for the bonus)
    float l_d;   // log2(1/S) of the draft row (mode 1)
    float c_hi, c_lo;
    int b;       // request
    int pad0;
    double u;    // sampling uniform
    double pad1;
};

struct Params {
    const char *tgt;
    const char *drf;
    const int32_t *tokens;
    const int32_t *verify_len;
    const float *temperature;
    unsigned long long seed;
    int B, K, V, nchunk, npart, nslot;
    int k0, k1;        // positions this wave verifies: [k0, k1) (one wave [0, K) unless early exit)
    int *ee_done;      // [B] request finished in an earlier wave (early exit), else null
    int32_t *out_tokens;
    int32_t *accept_len;
    uint32_t *dev_status;
    double *dbg_rows;  // [B, 2K+1, 2] or null
    double *dbg_probs; // [B, K, 2] or null
    // workspace
    ReqInfo *req;
    int *row_count;
    int4 *rows;        // (b, slot, greedy, log2(e)/T float bits) of every needed row, request-major
    float4 *part;      // [B, nslot, npart]: statistics-pass partials (one per 8 KiB item)
    float4 *sub;       // [B, nchunk]: sampler chunk masses A, B, W
    float4 *sexact;    // [B, nchunk]: exact sums of e (hi, lo) and e' (hi, lo)
    SampInfo *samp_list; // [B] one record per sampled request, in request order
    int *samp_count;     // number of sampled requests (records in samp_list), from sv_prep
    // confidence-scheduled verification (spec_verify_scheduled)
    const float *sched_mp;  // [B, K] draft max-probabilities: sv_prep takes L from the
                            // threshold schedule of these (verify_len unused), or null
    float sched_thr;        // the schedule's threshold
    int32_t *vlen_out;      // [B] the scheduled lengths, written by sv_prep (nullable)
    int draft_ready;        // the draft rows' partials are already in `part` (a confidence
                            // pass over the same rows at the same T): list target rows only
    // LM-head path (spec_verify_lmhead): the logits exist only inside the GEMM
    const float *gz;        // [B, nslot] logit of each row at its draft token, or null
    const char *samp_t;     // fp32 rows: list entry li's target draw row at samp_t + li * samp_stride rows
    const char *samp_d;     // and its draft row (residual draws) at samp_d + li * samp_stride rows
    int samp_stride;
};

__device__ __forceinline__ const char *row_ptr(const Params &P, int b, int slot, int esz) {
    if (slot <= P.K)
        return P.tgt + ((size_t)b * (size_t)(P.K + 1) + (size_t)slot) * (size_t)P.V * esz;
    return P.drf + ((size_t)b * (size_t)P.K + (size_t)(slot - P.K - 1)) * (size_t)P.V * esz;
}

// Row of a sampled request's draw: list entry li's recomputed row on the
// LM-head path, else the request's logit row.
__device__ __forceinline__ const char *samp_row(const Params &P, int li, int b, int slot, int esz,
                                                bool draft) {
    if (P.samp_t)
        return (draft ? P.samp_d : P.samp_t) + (size_t)li * (size_t)P.samp_stride * (size_t)P.V * esz;
    return row_ptr(P, b, slot, esz);
}

__device__ __forceinline__ float load_logit(const char *row, int dt, int x) {
    if (dt == kBF16) {
        uint16_t h = __ldg(reinterpret_cast<const uint16_t *>(row) + x);
        return __uint_as_float((uint32_t)h << 16);
    }
    return __ldg(reinterpret_cast<const float *>(row) + x);
}

// ------------------------------------------------------------------ 1. prep

// Rows a request needs in the wave of positions [k0, k1): target rows k0..t1
// (t1 = L when L <= k1, the bonus / last row, else k1 - 1) and, when sampled,
// draft rows k0..min(k1, L) - 1.  Returns the count; row r has slot
// wave_slot(r, ...).  With one wave [0, K) this is every row of the request.
__device__ __forceinline__ int wave_rows(int L, bool greedy, int k0, int k1, int &nt) {
    const int t1 = L <= k1 ? L : k1 - 1;
    nt = max(t1 - k0 + 1, 0);
    const int nd = greedy ? 0 : max(min(k1, L) - k0, 0);
    return nt + nd;
}
__device__ __forceinline__ int wave_slot(int r, int nt, int k0, int K) {
    return r < nt ? k0 + r : K + 1 + k0 + (r - nt);
}

// log2(e)/T of a sampled request: c = fl(log2(e)/T) (the statistics pass's
// factor) and the same value as c_hi + c_lo: c_hi = fl(hi/T), its exact
// remainder, then the low part, with the high part kept at or below the value
// and the low part positive.
__device__ __forceinline__ void temp_coeffs(float T, float &c, float &c_hi, float &c_lo) {
    const float q = __fdiv_rn(kLog2EHi, T);
    const float rem = __fmaf_rn(-q, T, kLog2EHi);
    float ql = __fdiv_rn(__fadd_rn(rem, kLog2ELo), T);
    float chi = q;
    if (ql < 0.f) {
        chi = __int_as_float(__float_as_int(q) - 1);
        ql = __fadd_rn(ql, __fsub_rn(q, chi));
    }
    if (!(ql >= FLT_MIN)) ql = FLT_MIN;
    c = q;
    c_hi = chi;
    c_lo = ql;
}

// Threshold schedule of one request: the longest prefix whose fp32 running
// product of draft max-probabilities, multiplied left to right, stays at or
// above thr.  The row is loaded whole first (independent loads), then the
// product runs on registers in the same order.
__device__ __forceinline__ int schedule_threshold(const float *mp, int K, float thr) {
    float v[SPEC_MAX_K];
#pragma unroll
    for (int k = 0; k < SPEC_MAX_K; ++k) v[k] = k < K ? __ldg(mp + k) : 0.f;
    float prod = 1.0f;
    int L = 0;
    bool run = true;
#pragma unroll
    for (int k = 0; k < SPEC_MAX_K; ++k) {
        if (run && k < K) {
            prod = __fmul_rn(prod, v[k]);
            if (prod >= thr) L = k + 1;
            else run = false;
        }
    }
    return L;
}

constexpr int kPrepThreads = 1024;
// Threads of the per-batch set-up kernel for B requests: one per request up to
// kPrepThreads (each thread adds the warp totals before its own, so a block
// no larger than the batch keeps that short).
static inline int prep_threads(int B) { return B >= kPrepThreads ? kPrepThreads : ((B + 31) / 32) * 32; }
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded wait: 2 s
// Diagnostics: the DIAG instantiations of the bulk-copy kernels (launched only
// while the switch is on) make every warp first wait on a barrier nothing
// completes; that wait runs out after kDiagWaitNs and the warp gives up as on
// a real timeout (status bit, its copies drained, no items).
static bool g_diag_timeout = false;
constexpr unsigned long long kDiagWaitNs = 1000000ull;  // 1 ms

// The diagnostic wait of one warp: true when the warp must give up.
__device__ __forceinline__ bool diag_wait_runs_out(uint64_t *never) {
    return !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(never, 0u, kDiagWaitNs));
}

__global__ void __launch_bounds__(kPrepThreads) sv_prep(Params P) {
    __shared__ int warp_tot[kPrepThreads / 32], warp_smp[kPrepThreads / 32];
    __shared__ int carry_s, carry_o;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nthr = blockDim.x, nw = nthr >> 5;  // a multiple of 32, at most kPrepThreads
    if (tid == 0) {
        carry_s = 0;
        carry_o = 0;
    }
    __syncthreads();
    pdl_trigger();
    const bool first_wave = P.k0 == 0;
    for (int base = 0; base < P.B; base += nthr) {
        const int b = base + tid;
        int n = 0, L = 0, greedy = 1, nt = 0, smp = 0;
        float cval = 0.f;
        ReqInfo ri;
        if (b < P.B && !first_wave) {  // a later wave: the records exist, finished requests drop out
            ri = P.req[b];
            L = ri.L;
            greedy = ri.greedy;
            cval = ri.c;
            n = P.ee_done[b] ? 0 : wave_rows(L, greedy != 0, P.k0, P.k1, nt);
        } else if (b < P.B) {
            uint32_t st = 0;
            if (P.sched_mp) {  // threshold schedule: fp32 running product, left to right
                L = schedule_threshold(P.sched_mp + (size_t)b * P.K, P.K, P.sched_thr);
                if (P.vlen_out) P.vlen_out[b] = L;
            } else {
                L = P.verify_len ? P.verify_len[b] : P.K;
            }
            const float T = P.temperature[b];
            if (L < 0) { L = 0; st |= SPEC_DEV_BAD_LEN; }
            if (L > P.K) { L = P.K; st |= SPEC_DEV_BAD_LEN; }
            // (a draft token outside [0, V) cuts the length further; sv_decide
            // applies that cut, so the rows listed here may include a few the
            // step then ignores, and this kernel, which the statistics pass
            // waits for, loads no tokens)
            greedy = !(isfinite(T) && T >= FLT_MIN);
            smp = greedy ? 0 : 1;
            ri.L = L;
            ri.greedy = greedy;
            ri.T = T;
            if (!greedy) {
                temp_coeffs(T, ri.c, ri.c_hi, ri.c_lo);
            } else {
                ri.c = 0.f; ri.c_hi = 0.f; ri.c_lo = 0.f;
            }
            cval = ri.c;
            if (st && P.dev_status) atomicOr(P.dev_status, st);
            if (P.ee_done) P.ee_done[b] = 0;
            n = wave_rows(L, greedy != 0, P.k0, P.k1, nt);
            if (P.draft_ready) n = nt;  // draft partials exist: target rows only
        }
        // block exclusive scans of n (row-list offsets) and, in the first
        // wave, of the sampled flags (samp_list entries in request order)
        int incl = n, incl_o = smp;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            const int vo = __shfl_up_sync(0xFFFFFFFFu, incl_o, o);
            if (lane >= o) {
                incl += v;
                incl_o += vo;
            }
        }
        if (lane == 31) {
            warp_tot[w] = incl;
            warp_smp[w] = incl_o;
        }
        __syncthreads();
        int woff = 0, woff_o = 0, block_tot = 0, block_o = 0;
        for (int i = 0; i < nw; ++i) {
            if (i < w) {
                woff += warp_tot[i];
                woff_o += warp_smp[i];
            }
            block_tot += warp_tot[i];
            block_o += warp_smp[i];
        }
        const int off = carry_s + woff + incl - n;
        if (b < P.B) {
            if (first_wave) {
                ri.ord = smp ? carry_o + woff_o + incl_o - smp : -1;
                P.req[b] = ri;
            }
            for (int r = 0; r < n; ++r)
                P.rows[off + r] = make_int4(b, wave_slot(r, nt, P.k0, P.K), greedy, __float_as_int(cval));
        }
        __syncthreads();
        if (tid == 0) {
            carry_s += block_tot;
            carry_o += block_o;
        }
        __syncthreads();
    }
    if (tid == 0) {
        *P.row_count = carry_s;
        if (first_wave) *P.samp_count = carry_o;
    }
}

// ------------------------------------------------------------------ 2. statistics pass

constexpr int kP1Warps = 4;          // warps per CTA (two CTAs per SM); each runs its own copy ring
constexpr int kStages = 3;           // bulk-copy stages per warp
constexpr int kP1ItemBytes = 8192;   // logits per item (one bulk copy, one partial)
constexpr int kSubVecs = 256;        // 16-byte vectors per 4 KiB sub-block (8 per lane)
constexpr int kP1Vecs = kP1ItemBytes / 16;
template <int DT> __host__ __device__ constexpr int p1_item_elems() {
    return kP1ItemBytes / Fmt<DT>::kESZ;
}

// What the issuing lane learned about a stage's item (the consumer reads it
// from shared memory instead of global metadata).
struct StageDesc {
    int b, slot, c, nvec;
    float cval;
    int greedy;
    int pad0, pad1;
};

struct P1Shared {
    uint4 buf[kP1Warps][kStages][kP1Vecs];
    StageDesc desc[kP1Warps][kStages];
    unsigned long long bar[kP1Warps][kStages];
    unsigned long long never[kP1Warps];  // diagnostics: a barrier nothing completes
};

// Lane maximum of 8 vectors (vectors at or past nvec - q0 excluded unless FULL).
template <int DT, bool FULL>
__device__ __forceinline__ float lane_max8(const uint4 (&v)[8], int lim, int lane) {
    float lm = -INFINITY;
    if (DT == kBF16) {
        uint32_t run = 0xFF80FF80u;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (FULL || i * 32 + lane < lim)
                run = bf16x2_max(run, bf16x2_max(bf16x2_max(v[i].x, v[i].y), bf16x2_max(v[i].z, v[i].w)));
        lm = fmaxf(__uint_as_float(run << 16), __uint_as_float(run & 0xFFFF0000u));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (FULL || i * 32 + lane < lim) lm = fmaxf(lm, vec_max<DT>(v[i]));
    }
    return lm;
}

// Sum of 2^((z - m) c) over the lane's elements of 8 vectors.
template <int DT, bool FULL>
__device__ __forceinline__ float lane_expsum8(const uint4 (&v)[8], int lim, float m, float c,
                                              int lane) {
    const unsigned long long m2 = f2u(make_float2(m, m)), c2 = f2u(make_float2(c, c));
    unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (FULL || i * 32 + lane < lim) {
            if (DT == kBF16) {
                bf16x2_exp_acc(v[i].x, m2, c2, a0);
                bf16x2_exp_acc(v[i].y, m2, c2, a1);
                bf16x2_exp_acc(v[i].z, m2, c2, a0);
                bf16x2_exp_acc(v[i].w, m2, c2, a1);
            } else {
                f32x2_exp_acc(v[i].x, v[i].y, m2, c2, a0);
                f32x2_exp_acc(v[i].z, v[i].w, m2, c2, a1);
            }
        }
    }
    const float2 t = add2(u2f(a0), u2f(a1));
    return t.x + t.y;
}

// Offset (in elements from the sub-block start) of the lane's first element
// equal to x, or INT_MAX.  Compares raw bit patterns (x is one of the
// elements), with +0 and -0 treated as equal as floats compare them.
template <int DT, bool FULL>
__device__ __forceinline__ int first_equal8(const uint4 (&v)[8], int lim, float x, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    int off = INT_MAX;
    if (DT == kBF16) {
        const uint32_t key = __float_as_uint(x) >> 16;
        const uint32_t msk = (key & 0x7FFFu) == 0 ? 0x7FFF7FFFu : 0xFFFFFFFFu;
        const uint32_t key2 = (key | (key << 16)) & msk;
#pragma unroll
        for (int i = 7; i >= 0; --i) {  // the last hit written is the lowest index
            if (FULL || i * 32 + lane < lim) {
                const uint32_t m0 = __vcmpeq2(v[i].x & msk, key2), m1 = __vcmpeq2(v[i].y & msk, key2);
                const uint32_t m2 = __vcmpeq2(v[i].z & msk, key2), m3 = __vcmpeq2(v[i].w & msk, key2);
                const uint32_t bits = (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) |
                                      ((m2 & 1u) << 4) | ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) |
                                      ((m3 >> 9) & 128u);
                if (bits) off = (i * 32 + lane) * EPV + (__ffs(bits) - 1);
            }
        }
    } else {
        const uint32_t key = __float_as_uint(x);
        const uint32_t msk = (key & 0x7FFFFFFFu) == 0 ? 0x7FFFFFFFu : 0xFFFFFFFFu;
        const uint32_t k2 = key & msk;
#pragma unroll
        for (int i = 7; i >= 0; --i) {
            if (FULL || i * 32 + lane < lim) {
                const uint32_t bits = ((v[i].x & msk) == k2 ? 1u : 0u) | ((v[i].y & msk) == k2 ? 2u : 0u) |
                                      ((v[i].z & msk) == k2 ? 4u : 0u) | ((v[i].w & msk) == k2 ? 8u : 0u);
                if (bits) off = (i * 32 + lane) * EPV + (__ffs(bits) - 1);
            }
        }
    }
    return off;
}

// Lane-local running statistics over the 4 KiB sub-blocks of one item: sampled
// rows keep (max, sum 2^((z - max) c)) rescaled when the max grows; greedy rows
// keep (max, lowest index of it).  The lane's elements come in increasing index
// order (vector i * 32 + lane of each sub-block, sub-blocks in order).
struct LaneStat {
    float m, s;
    int idx;
};

template <int DT, bool FULL>
__device__ __forceinline__ void lane_update(LaneStat &st, const uint4 (&v)[8], int lim, bool greedy,
                                            float c, int e_base, int lane) {
    const float lm = lane_max8<DT, FULL>(v, lim, lane);
    if (greedy) {
        if (lm > st.m || (st.idx == INT_MAX && lm == st.m && lim > 0)) {  // also an all -inf start
            st.m = lm;
            const int j = first_equal8<DT, FULL>(v, lim, lm, lane);
            st.idx = j == INT_MAX ? INT_MAX : e_base + j;
        }
        return;
    }
    if (lm > st.m) {
        if (st.m > -INFINITY) st.s *= ex2((st.m - lm) * c);
        st.m = lm;
    }
    if (st.m > -INFINITY) st.s += lane_expsum8<DT, FULL>(v, lim, st.m, c, lane);
}

// Warp-wide partial of an item from the lanes' statistics: greedy rows
// {max, -, lowest argmax, -}; sampled rows {max, sum 2^((z - max) c), -1, -}.
__device__ __forceinline__ float4 warp_partial(const LaneStat &st, bool greedy, float c) {
    const float m = warp_max(st.m);
    if (greedy) return make_float4(m, 0.f, __int_as_float(warp_min_int(st.m == m ? st.idx : INT_MAX)), 0.f);
    const float s = (st.m > -INFINITY) ? st.s * ex2((st.m - m) * c) : 0.f;
    return make_float4(m, warp_sum(s), __int_as_float(-1), 0.f);
}

// One item = 8 KiB of one needed logit row (one partial per item); item k of
// a warp is first + k * total_warps (request-major order across the grid).
// Each warp keeps kStages bulk copies in flight into its own shared-memory
// ring and reads each stage in 4 KiB sub-blocks; the row metadata of 32 items
// at a time is gathered across the lanes, so neither the issue nor the
// consumption of an item waits on a global load.
template <int DT, bool VEC, bool DIAG = false>
__global__ void __launch_bounds__(kP1Warps * 32, 1) sv_pass1(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = p1_item_elems<DT>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    P1Shared &sh = *reinterpret_cast<P1Shared *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4(*buf)[kP1Vecs] = sh.buf[warp];
    StageDesc *desc = sh.desc[warp];
    unsigned long long *bar = sh.bar[warp];
    if (VEC && lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(reinterpret_cast<uint64_t *>(&bar[s]), 1);
        mbar_init(reinterpret_cast<uint64_t *>(&sh.never[warp]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_wait();  // the row list comes from sv_prep
    pdl_trigger();
    const uint32_t nitems = (uint32_t)(*P.row_count) * (uint32_t)P.npart;
    const uint32_t first = blockIdx.x * kP1Warps + warp;
    const uint32_t stride = gridDim.x * kP1Warps;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const uint4 neg_inf = make_uint4(ni, ni, ni, ni);

    // per-lane metadata of the warp's items [mk0, mk0 + 32)
    int4 mrow = make_int4(0, 0, 0, 0);
    uint32_t mc = 0;
    uint32_t mk0 = 0x80000000u;  // no window yet (item counts stay below 2^31)
    auto meta = [&](uint32_t k, int4 &r, uint32_t &c) {
        if (k - mk0 >= 32u) {  // gather the next 32 items' metadata
            mk0 = k & ~31u;
            const uint32_t item = first + (mk0 + (uint32_t)lane) * stride;
            if (item < nitems) {
                const uint32_t ri = item / (uint32_t)P.npart;
                mc = item - ri * (uint32_t)P.npart;
                mrow = P.rows[ri];
            }
        }
        const int j = (int)(k - mk0);
        r.x = __shfl_sync(0xFFFFFFFFu, mrow.x, j);
        r.y = __shfl_sync(0xFFFFFFFFu, mrow.y, j);
        r.z = __shfl_sync(0xFFFFFFFFu, mrow.z, j);
        r.w = __shfl_sync(0xFFFFFFFFu, mrow.w, j);
        c = __shfl_sync(0xFFFFFFFFu, mc, j);
    };
    const uint32_t nk = (nitems > first) ? (nitems - first + stride - 1) / stride : 0u;

    // issue item k of this warp into stage k % kStages
    auto issue = [&](uint32_t k) {
        int4 r;
        uint32_t c;
        meta(k, r, c);
        if (lane == 0) {
            const int s = (int)(k % kStages);
            const uint32_t e0 = c * CE;
            const uint32_t bytes = min((uint32_t)CE, (uint32_t)P.V - e0) * ESZ;
            StageDesc d;
            d.b = r.x; d.slot = r.y; d.c = (int)c; d.nvec = (int)(bytes / 16);
            d.cval = __int_as_float(r.w); d.greedy = r.z; d.pad0 = d.pad1 = 0;
            desc[s] = d;
            fence_proxy_async();  // the stage's previous contents were read by this warp
            mbar_expect_tx(reinterpret_cast<uint64_t *>(&bar[s]), bytes);
            bulk_g2s(buf[s], row_ptr(P, r.x, r.y, ESZ) + (size_t)e0 * ESZ, bytes,
                     reinterpret_cast<uint64_t *>(&bar[s]));
        }
        __syncwarp();
    };

    if (VEC)
        for (uint32_t k = 0; k < (uint32_t)kStages && k < nk; ++k) issue(k);
    uint32_t k = 0;
    bool failed = false;
    if (VEC && DIAG) failed = diag_wait_runs_out(reinterpret_cast<uint64_t *>(&sh.never[warp]));
    if (!failed) for (; k < nk; ++k) {
        LaneStat st{-INFINITY, 0.f, INT_MAX};
        StageDesc d;
        if (VEC) {
            const int s = (int)(k % kStages);
            const bool ok = mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[s]), (k / kStages) & 1u,
                                              kWaitLimitNs);
            if (!__all_sync(0xFFFFFFFFu, ok)) {  // the warp gives up together
                failed = true;
                break;
            }
            d = desc[s];
            const bool greedy = d.greedy != 0;
            const int e0 = d.c * CE;
            if (d.nvec == kP1Vecs) {
#pragma unroll
                for (int sb = 0; sb < kP1Vecs / kSubVecs; ++sb) {
                    uint4 v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = buf[s][sb * kSubVecs + i * 32 + lane];
                    lane_update<DT, true>(st, v, kSubVecs, greedy, d.cval, e0 + sb * kSubVecs * EPV, lane);
                }
            } else {
                for (int sb = 0; sb * kSubVecs < d.nvec; ++sb) {
                    uint4 v[8];
                    const int lim = d.nvec - sb * kSubVecs;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v[i] = i * 32 + lane < lim ? buf[s][sb * kSubVecs + i * 32 + lane] : neg_inf;
                    lane_update<DT, false>(st, v, lim, greedy, d.cval, e0 + sb * kSubVecs * EPV, lane);
                }
            }
            __syncwarp();
            if (k + kStages < nk) issue(k + kStages);
        } else {
            int4 r;
            uint32_t c;
            meta(k, r, c);
            d.b = r.x; d.slot = r.y; d.c = (int)c; d.cval = __int_as_float(r.w); d.greedy = r.z;
            const int e0 = (int)(c * CE);
            const int nvec = (int)((min((uint32_t)CE, (uint32_t)P.V - (uint32_t)e0) + EPV - 1) / EPV);
            const char *row = row_ptr(P, r.x, r.y, ESZ);
            for (int sb = 0; sb * kSubVecs < nvec; ++sb) {
                uint4 v[8];
                const int lim = nvec - sb * kSubVecs;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = load_vec<DT, false>(row, (long long)e0 + (long long)(sb * kSubVecs + i * 32 + lane) * EPV, P.V);
                lane_update<DT, false>(st, v, lim, d.greedy != 0, d.cval, e0 + sb * kSubVecs * EPV, lane);
            }
        }
        const float4 out = warp_partial(st, d.greedy != 0, d.cval);
        if (lane == 0) P.part[((size_t)d.b * P.nslot + d.slot) * P.npart + d.c] = out;
    }
    if (VEC && failed) {
        // report, then let every copy this warp still has in flight land
        if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        for (uint32_t kk = k; kk < k + kStages && kk < nk; ++kk)
            mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[kk % kStages]), (kk / kStages) & 1u,
                              kWaitLimitNs);
    }
}

// ------------------------------------------------------------------ 3. decide

constexpr int kPerLane = 4;      // chunk records held in registers per lane (128 per warp)
// rows whose chunk records one warp loads at once: 5 (8 warps cover K = 16's
// 33 rows in one round) at the compiler's register budget, 3 in the build cut
// to 64 registers
template <int MINB> __host__ __device__ constexpr int rows_per_warp() { return MINB >= 4 ? 3 : 5; }

// Row statistics from one block of up to 32 * kPerLane chunk records held by
// the warp: {max, S (sampled rows), lowest argmax bits (greedy rows)}.
__device__ __forceinline__ void reduce_block(const float4 (&q)[kPerLane], bool greedy, float c,
                                             float &m, float &S, int &amax) {
    float mr = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) mr = fmaxf(mr, q[i].x);
    mr = warp_max(mr);
    if (greedy) {
        int ar = INT_MAX;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            if (q[i].x == mr) ar = min(ar, __float_as_int(q[i].z));
        ar = warp_min_int(ar);
        if (mr > m || (mr == m && ar < amax)) amax = ar;
        m = fmaxf(m, mr);
    } else {
        const float mn = fmaxf(m, mr);
        float Sr = 0.f;
        if (mn > -INFINITY) {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (q[i].x > -INFINITY) Sr += q[i].y * ex2((q[i].x - mn) * c);
            if (m > -INFINITY) S *= ex2((m - mn) * c);
        }
        S += warp_sum(Sr);
        m = mn;
    }
}

__device__ __forceinline__ float4 part_filler() {
    return make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
}

// Row statistics of any chunk count (one warp, blocks of 32 * kPerLane).
__device__ __forceinline__ float4 combine_row(const Params &P, int b, int slot, bool greedy,
                                              float c, int lane) {
    const float4 *pp = P.part + ((size_t)b * P.nslot + slot) * P.npart;
    const int n = P.npart;
    float m = -INFINITY, S = 0.f;
    int amax = INT_MAX;
    for (int base = 0; base < n; base += 32 * kPerLane) {
        float4 q[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int ci = base + i * 32 + lane;
            q[i] = ci < n ? pp[ci] : part_filler();
        }
        reduce_block(q, greedy, c, m, S, amax);
    }
    return make_float4(m, S, __int_as_float(amax), 0.f);
}


// Acceptance test u * q(x) < p(x) of one position, as u < p/q with
// p/q = 2^(((g - m) - (g' - m')) c) * S'/S; the exponent is formed in
// two-float arithmetic so that the ratio carries only the float error of the
// row sums and of ex2.
__device__ __forceinline__ bool accept_position(float u, float g, float m_t, float S_t, float gd,
                                                float m_d, float S_d, float c_hi, float c_lo) {
    if (!(S_t > 0.f) || g == -INFINITY) return false;  // p = 0
    if (!(S_d > 0.f) || gd == -INFINITY) return true;   // q = 0 < p
    if (u == 0.f) return true;                          // 0 < p
    const FF dt = two_sum(g, -m_t), dd = two_sum(gd, -m_d);
    const FF D = ff_add(dt, FF{-dd.hi, -dd.lo});
    const float th = __fmul_rn(D.hi, c_hi);
    if (th > 128.f) return true;    // ratio above 2^127 > u
    if (th < -160.f) return false;  // ratio below 2^-159 < 2^-24 <= u
    const float tl = __fadd_rn(__fmaf_rn(D.hi, c_hi, -th), __fmaf_rn(D.hi, c_lo, __fmul_rn(D.lo, c_hi)));
    const float r = __fmul_rn(__fmul_rn(ex2(th), __fmaf_rn(tl, kLn2F, 1.f)), __fdiv_rn(S_d, S_t));
    return u < r;
}

// MINB: CTAs per SM the register budget is cut for (0: the compiler's own
// budget; 4 when the batch would not fit one wave at that budget).
template <int DT, int MINB = 0>
__global__ void __launch_bounds__(kThreads, MINB) sv_decide(Params P) {
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = P.K;
    __shared__ float s_m[2 * SPEC_MAX_K + 1];
    __shared__ float s_S[2 * SPEC_MAX_K + 1];
    __shared__ int s_amax[SPEC_MAX_K + 1];
    __shared__ int s_a;
    // inputs and sv_prep's results (two kernels back) may be read before the wait
    const ReqInfo rq = P.req[b];
    const bool greedy = rq.greedy != 0;
    // the first draft token outside [0, V) cuts the verify length (every warp
    // forms the cut itself from the tokens; the status bit from warp 0)
    const int x = lane < rq.L ? P.tokens[(size_t)b * K + lane] : 0;
    const unsigned bad = __ballot_sync(0xFFFFFFFFu, lane < rq.L && (x < 0 || x >= P.V));
    const int L = bad ? __ffs(bad) - 1 : rq.L;
    if (bad && tid == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_BAD_TOKEN);
    float g = 0.f, gd = 0.f, u = 0.f;
    // the sampling uniform of every position the emitted token may take
    // (lane k: position k), drawn before the wait
    const double us_lane = (warp == 0 && !greedy && lane <= L) ? uniform_sample(P.seed, (uint32_t)b,
                                                                               (uint32_t)lane)
                                                              : 0.0;
    if (warp == 0 && lane < L) {
        if (!greedy) {
            if (!P.gz) {
                g = load_logit(row_ptr(P, b, lane, Fmt<DT>::kESZ), DT, x);
                gd = load_logit(row_ptr(P, b, K + 1 + lane, Fmt<DT>::kESZ), DT, x);
            }
            u = uniform_accept_f(P.seed, (uint32_t)b, (uint32_t)lane);
        }
    }
    pdl_wait();  // chunk partials come from sv_pass1
    pdl_trigger();
    if (P.gz && warp == 0 && lane < L && !greedy) {  // written by the LM-head GEMM's epilogue
        g = P.gz[(size_t)b * P.nslot + lane];
        gd = P.gz[(size_t)b * P.nslot + K + 1 + lane];
    }
    if (P.ee_done && P.ee_done[b]) return;  // finished in an earlier wave (uniform over the CTA)
    // the rows of this wave: positions [k0, e) and, when L <= k1, the row L
    const int k0 = P.k0, e = min(P.k1, L);
    int nt;
    const int nrows = wave_rows(L, greedy, k0, P.k1, nt);
    if (P.npart <= 32 * kPerLane) {
        // each warp loads the records of up to RPW rows, then reduces them
        constexpr int RPW = rows_per_warp<MINB>();
        for (int r0 = warp; r0 < nrows; r0 += kWarps * RPW) {
            float4 q[RPW][kPerLane];
#pragma unroll
            for (int j = 0; j < RPW; ++j) {
                const int r = r0 + j * kWarps;
                const float4 *pp =
                    P.part + ((size_t)b * P.nslot + wave_slot(r < nrows ? r : 0, nt, k0, K)) * P.npart;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    const int ci = i * 32 + lane;
                    q[j][i] = (r < nrows && ci < P.npart) ? pp[ci] : part_filler();
                }
            }
#pragma unroll
            for (int j = 0; j < RPW; ++j) {
                const int r = r0 + j * kWarps;
                if (r < nrows) {
                    float m = -INFINITY, S = 0.f;
                    int amax = INT_MAX;
                    reduce_block(q[j], greedy, rq.c, m, S, amax);
                    const int slot = wave_slot(r, nt, k0, K);
                    if (lane == 0) {
                        s_m[slot] = m;
                        s_S[slot] = S;
                        if (slot <= K) s_amax[slot] = amax;
                    }
                }
            }
        }
    } else {
        for (int r = warp; r < nrows; r += kWarps) {
            const int slot = wave_slot(r, nt, k0, K);
            const float4 rs = combine_row(P, b, slot, greedy, rq.c, lane);
            if (lane == 0) {
                s_m[slot] = rs.x;
                s_S[slot] = rs.y;
                if (slot <= K) s_amax[slot] = __float_as_int(rs.z);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        bool acc = true;  // positions before k0 were accepted in earlier waves
        if (lane >= k0 && lane < e) {
            if (greedy)
                acc = (x == s_amax[lane]);
            else
                acc = accept_position(u, g, s_m[lane], s_S[lane], gd, s_m[K + 1 + lane],
                                      s_S[K + 1 + lane], rq.c_hi, rq.c_lo);
        }
        if (P.dbg_probs && lane < K) {
            double p = NAN, q = NAN;
            if (!greedy && lane < L) {
                const double cd = kLog2E / (double)rq.T;
                const float St = s_S[lane], Sd = s_S[K + 1 + lane];
                p = St > 0.f ? exp2(((double)g - (double)s_m[lane]) * cd) / (double)St : 0.0;
                q = Sd > 0.f ? exp2(((double)gd - (double)s_m[K + 1 + lane]) * cd) / (double)Sd : 0.0;
            }
            P.dbg_probs[((size_t)b * K + lane) * 2 + 0] = p;
            P.dbg_probs[((size_t)b * K + lane) * 2 + 1] = q;
        }
        const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc);
        // first rejection; with none, the request ends at L if this wave
        // listed target row L (the last row sv_prep listed is t1, from the
        // length before the bad-token cut), else it stays open for the next
        // wave (-1)
        const int t1 = rq.L <= P.k1 ? rq.L : P.k1 - 1;
        const int a = rej ? min(__ffs(rej) - 1, L) : (L <= t1 ? L : -1);
        if (lane == 0) s_a = a;
    }
    __syncthreads();
    const int a = s_a;
    if (a < 0) return;  // uniform over the CTA
    const double ua = __shfl_sync(0xFFFFFFFFu, us_lane, a & 31);  // position a's (a <= 31)
    if (P.ee_done && threadIdx.x == 0) P.ee_done[b] = 1;
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    for (int k = tid; k <= K; k += kThreads) {
        int v = -1;
        if (k < a) v = x;  // thread k < a <= L is lane k of warp 0, which holds draft token k
        else if (k == a && greedy) v = s_amax[a];
        out[k] = v;
    }
    if (tid == 0) {
        P.accept_len[b] = a;
        if (!greedy) {
            SampInfo si;
            si.mode = a < L ? 1 : 2;
            si.a = a;
            si.slot_t = a;
            si.slot_d = K + 1 + a;
            si.m_t = s_m[a];
            si.l_t = 0.f;
            si.m_d = 0.f;
            si.l_d = 0.f;
            if (si.mode == 1) {  // any constant factor cancels against the exact sums
                si.l_t = -__log2f(s_S[a]);
                si.m_d = s_m[K + 1 + a];
                si.l_d = -__log2f(s_S[K + 1 + a]);
            }
            si.c_hi = rq.c_hi;
            si.c_lo = rq.c_lo;
            si.b = b;
            si.pad0 = 0;
            si.u = a < 32 ? ua : uniform_sample(P.seed, (uint32_t)b, (uint32_t)a);
            si.pad1 = 0.0;
            P.samp_list[rq.ord] = si;
        }
    }
    if (P.dbg_rows) {
        const int nslot = 2 * K + 1;
        for (int sl = tid; sl < nslot; sl += kThreads) {
            double m = NAN, ls = NAN;
            if (!greedy && (sl <= L || (sl >= K + 1 && sl - K - 1 < L))) {
                m = (double)s_m[sl] / (double)rq.T;
                ls = log((double)s_S[sl]);
            }
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 0] = m;
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 1] = ls;
        }
    }
}

// ------------------------------------------------------------------ 4. sampler pass

// Masses of one 4 KiB chunk of the sampled row (pair).  Per element pair
// (target z, draft z'): a = 2^((z - m) c + l), b = 2^((z' - m') c + l') with
// the row maxima, the two-float c and l = log2(1/S) from the statistics pass.
// Over {a > b}: D = sum of (a - b) and Bm = sum of b (warp totals).  The
// element weights are also added exactly (Fast2Sum against a biased
// accumulator) into `acc`, whose totals over the whole row give the exact
// normalisers sum a, sum b.  With kappa = 1 / (sum a) = 1 + delta, a chunk's
// residual mass is kappa A - kappa' Bm = D + delta (D + Bm) - delta' Bm,
// A = D + Bm; for the bonus (b = 0) D is the chunk's mass of p.
template <int DT>
__device__ __forceinline__ void sample_masses(const uint4 (&vt)[kVecPerLane],
                                              const uint4 (&vd)[kVecPerLane], int nvec,
                                              const SampInfo &si, float &D, float &Bm,
                                              BiasAcc2 &acc, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    const float2 m2 = make_float2(si.m_t, si.m_d);
    const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
    const float2 l2 = make_float2(si.l_t, si.l_d);
    D = 0.f; Bm = 0.f;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) {
        if (i * 32 + lane < nvec) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const float2 ab = weight2l(make_float2(elem<DT>(vt[i], e), elem<DT>(vd[i], e)), m2, chi2, clo2, l2);
                acc.add(ab);
                if (ab.x > ab.y) {
                    D = __fadd_rn(D, __fsub_rn(ab.x, ab.y));
                    Bm = __fadd_rn(Bm, ab.y);
                }
            }
        }
    }
    D = warp_sum(D);
    Bm = warp_sum(Bm);
}

constexpr int kSWarps = 2;      // warps per CTA of the sampler pass
constexpr int kSStages = 1;     // stages per warp; a stage holds a target and a draft chunk
constexpr int kSMinBlocks = 8;  // CTAs per SM the register budget is cut for (16 warps)

struct SShared {
    uint4 buf[kSWarps][kSStages][2 * kChunkBytes / 16];
    SampInfo info[kSWarps][kSStages];
    int item_b[kSWarps][kSStages], item_c[kSWarps][kSStages], item_nvec[kSWarps][kSStages];
    unsigned long long bar[kSWarps][kSStages];
    unsigned long long never[kSWarps];  // diagnostics: a barrier nothing completes
};

// Items = (sampled request, 4 KiB chunk) over the list sv_decide built (in
// request order), request-major; warp w takes the contiguous range
// [w n / W, (w + 1) n / W), so it changes request (and reloads the request's
// SampInfo) at most a few times.  Per item it writes the chunk's {D, Bm}; the
// exact sums are written once per (warp, request) segment, at the segment's
// last chunk, with zeros at the others.  Same per-warp ring as sv_pass1.
template <int DT, bool VEC, bool DIAG = false>
__global__ void __launch_bounds__(kSWarps * 32, kSMinBlocks) sv_sample(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = chunk_elems<DT>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    SShared &sh = *reinterpret_cast<SShared *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long *bar = sh.bar[warp];
    if (VEC && lane == 0) {
        for (int s = 0; s < kSStages; ++s) mbar_init(reinterpret_cast<uint64_t *>(&bar[s]), 1);
        mbar_init(reinterpret_cast<uint64_t *>(&sh.never[warp]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_wait();  // the sampled-request list and SampInfo come from sv_decide
    pdl_trigger();
    const uint64_t nitems = (uint64_t)(*P.samp_count) * (uint64_t)P.nchunk;
    const uint64_t nw = (uint64_t)gridDim.x * kSWarps;
    const uint64_t gw = (uint64_t)blockIdx.x * kSWarps + warp;
    const uint32_t k_begin = (uint32_t)(nitems * gw / nw);
    const uint32_t nk = (uint32_t)(nitems * (gw + 1) / nw) - k_begin;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const uint4 neg_inf = make_uint4(ni, ni, ni, ni);

    // request metadata of the current item (lane 0 only uses these in the ring)
    int cur_li = -1, cur_b = 0;
    SampInfo cur_si;
    auto item_of = [&](uint32_t k, uint32_t &c) {
        const uint32_t item = k_begin + k;
        const int li = (int)(item / (uint32_t)P.nchunk);
        c = item - (uint32_t)li * (uint32_t)P.nchunk;
        if (li != cur_li) {
            cur_li = li;
            cur_si = P.samp_list[li];
            cur_b = cur_si.b;
        }
    };
    auto issue = [&](uint32_t k) {
        if (lane == 0) {
            uint32_t c;
            item_of(k, c);
            const int s = (int)(k % kSStages);
            const uint32_t e0 = c * CE;
            const uint32_t bytes = min((uint32_t)CE, (uint32_t)P.V - e0) * ESZ;
            sh.info[warp][s] = cur_si;
            sh.item_b[warp][s] = cur_b;
            sh.item_c[warp][s] = (int)c;
            sh.item_nvec[warp][s] = (int)(bytes / 16);
            fence_proxy_async();
            uint64_t *fb = reinterpret_cast<uint64_t *>(&bar[s]);
            const bool two = cur_si.mode == 1;
            mbar_expect_tx(fb, two ? 2u * bytes : bytes);
            bulk_g2s(sh.buf[warp][s], samp_row(P, cur_li, cur_b, cur_si.slot_t, ESZ, false) + (size_t)e0 * ESZ,
                     bytes, fb);
            if (two)
                bulk_g2s(sh.buf[warp][s] + kChunkBytes / 16,
                         samp_row(P, cur_li, cur_b, cur_si.slot_d, ESZ, true) + (size_t)e0 * ESZ, bytes, fb);
        }
        __syncwarp();
    };
    if (VEC)
        for (uint32_t k = 0; k < (uint32_t)kSStages && k < nk; ++k) issue(k);
    FF seg_t{0.f, 0.f}, seg_d{0.f, 0.f};  // exact sums of the current request segment
    uint32_t k = 0;
    bool failed = false;
    if (VEC && DIAG) failed = diag_wait_runs_out(reinterpret_cast<uint64_t *>(&sh.never[warp]));
    if (!failed) for (; k < nk; ++k) {
        uint4 vt[kVecPerLane], vd[kVecPerLane];
        SampInfo si;
        int b, c, nvec;
        if (VEC) {
            const int s = (int)(k % kSStages);
            const bool ok = mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[s]),
                                              (k / kSStages) & 1u, kWaitLimitNs);
            if (!__all_sync(0xFFFFFFFFu, ok)) {  // the warp gives up together
                failed = true;
                break;
            }
            si = sh.info[warp][s];
            b = sh.item_b[warp][s];
            c = sh.item_c[warp][s];
            nvec = sh.item_nvec[warp][s];
            const bool resid = si.mode == 1;
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int q = i * 32 + lane;
                vt[i] = q < nvec ? sh.buf[warp][s][q] : neg_inf;
                vd[i] = (resid && q < nvec) ? sh.buf[warp][s][kChunkBytes / 16 + q] : neg_inf;
            }
            __syncwarp();
            if (k + kSStages < nk) issue(k + kSStages);
        } else {
            uint32_t cu;
            item_of(k, cu);  // every lane keeps its own copy here
            c = (int)cu;
            b = cur_b;
            si = cur_si;
            const long long e0 = (long long)c * CE;
            nvec = (int)((min((long long)CE, (long long)P.V - e0) + EPV - 1) / EPV);
            const bool resid = si.mode == 1;
            const char *rowt = samp_row(P, cur_li, b, si.slot_t, ESZ, false);
            const char *rowd = resid ? samp_row(P, cur_li, b, si.slot_d, ESZ, true) : rowt;
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const long long q = e0 + (long long)(i * 32 + lane) * EPV;
                vt[i] = load_vec<DT, false>(rowt, q, P.V);
                vd[i] = resid ? load_vec<DT, false>(rowd, q, P.V) : neg_inf;
            }
        }
        float Dm, Bm;
        BiasAcc2 acc;
        acc.init(1.0f);
        sample_masses<DT>(vt, vd, nvec, si, Dm, Bm, acc, lane);
        // fold the item's exact sums into the lane's two-float totals of this
        // request segment; the warp reduces them once, at the segment's end
        seg_t = ff_add(seg_t, FF{__fsub_rn(acc.h.x, 1.0f), acc.l.x});
        seg_d = ff_add(seg_d, FF{__fsub_rn(acc.h.y, 1.0f), acc.l.y});
        const bool seg_end = c == P.nchunk - 1 || k + 1 == nk;
        float4 ex = make_float4(0.f, 0.f, 0.f, 0.f);
        if (seg_end) {
            const FF st = warp_sum_ff(seg_t), sd = warp_sum_ff(seg_d);
            ex = make_float4(st.hi, st.lo, sd.hi, sd.lo);
            seg_t = FF{0.f, 0.f};
            seg_d = FF{0.f, 0.f};
        }
        if (lane == 0) {
            P.sub[(size_t)b * P.nchunk + c] = make_float4(Dm, Bm, 0.f, 0.f);
            P.sexact[(size_t)b * P.nchunk + c] = ex;  // nonzero only at a segment's last chunk
        }
    }
    if (VEC && failed) {
        if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        for (uint32_t kk = k; kk < k + kSStages && kk < nk; ++kk)
            mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[kk % kSStages]), (kk / kSStages) & 1u,
                              kWaitLimitNs);
    }
}

// ------------------------------------------------------------------ 5. inverse CDF

constexpr int kFindWarps = 4;  // warps per sampled request (one CTA each)
constexpr int kFindVecs = kChunkBytes / 16 / (kFindWarps * 32);  // chosen chunk's vectors per lane
static_assert(kFindVecs * kFindWarps * 32 * 16 == kChunkBytes, "the CTA covers the chunk");

// kappa - 1 for kappa = 1 / S, S a two-float sum close to 1.
__device__ __forceinline__ float kappa_minus_one(FF S) {
    return __fdiv_rn(__fsub_rn(__fsub_rn(1.f, S.hi), S.lo), S.hi);
}

// Scaled weights of one lane's 8 vectors of a chunk (lane-contiguous layout:
// vectors 8 * lane .. 8 * lane + 7), and the draw's weight of each element:
// the residual max(0, kappa a - kappa' b) or, from p, a.
template <int DT>
__device__ __forceinline__ float draw_weight(float2 ab, bool two, float dlt, float dld) {
    if (!two) return ab.x;
    return ab.x > ab.y ? fmaxf(0.f, __fadd_rn(__fsub_rn(ab.x, ab.y), __fmaf_rn(dlt, ab.x, -__fmul_rn(dld, ab.y))))
                       : 0.f;
}

// Token of one sampled request (one CTA), in float and two-float arithmetic
// (fp64 has a long dependent latency on this part).  Warp 0 picks the chunk:
// exact normalisers from the segment sums, chunk masses, a two-float prefix
// over the lanes (each lane owns a contiguous block of chunks).  Then every
// warp takes a contiguous slice of the chosen chunk (each lane kFindVecs
// contiguous vectors, lanes and warps in element order): the lane totals are
// scanned within the warp, the warp totals added in warp order, and the
// crossing lane walks its elements in order.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kFindWarps * 32) sv_find(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = chunk_elems<DT>();
    __shared__ int s_ch, s_two;
    __shared__ float s_th, s_dlt, s_dld;
    __shared__ float s_wt[kFindWarps];
    __shared__ int s_tok[kFindWarps], s_last[kFindWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the sampled-request list is sv_decide's (two kernels back, complete once
    // this kernel runs): read before the wait; the chunk masses come after it
    const int li = blockIdx.x;
    const bool active = li < *P.samp_count;  // uniform over the CTA
    SampInfo si;
    if (active) si = P.samp_list[li];
    pdl_wait();  // chunk masses come from sv_sample
    pdl_trigger();
    if (!active) return;
    const int b = si.b;
    const bool resid = si.mode == 1;
    const int nch = P.nchunk;
    float4 *sub = P.sub + (size_t)b * nch;
    const float4 *sex = P.sexact + (size_t)b * nch;
    const int per = (nch + 31) / 32;
    const int c0 = lane * per, c1 = min(nch, c0 + per);
    const bool held = per <= kPerLane;
    const char *rowt = samp_row(P, li, b, si.slot_t, ESZ, false);
    const char *rowd = resid ? samp_row(P, li, b, si.slot_d, ESZ, true) : rowt;
    const float2 m2 = make_float2(si.m_t, si.m_d);
    const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const uint4 neg_inf = make_uint4(ni, ni, ni, ni);

    if (warp == 0) {  // the chunk
        float4 q[kPerLane];
        float dlt = 0.f, dld = 0.f;
        if (held) {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) q[i] = c0 + i < c1 ? sub[c0 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (resid) {  // exact normalisers: sums over the segment records
            FF st{0.f, 0.f}, sd{0.f, 0.f};
            for (int c = c0; c < c1; ++c) {
                const float4 x = sex[c];
                st = ff_add(st, FF{x.x, x.y});
                sd = ff_add(sd, FF{x.z, x.w});
            }
            dlt = kappa_minus_one(warp_sum_ff(st));
            dld = kappa_minus_one(warp_sum_ff(sd));
        }
        // residual mass D + delta (D + Bm) - delta' Bm; the mass of p is D (bonus)
        auto mass_r = [&](const float4 &x) {
            return fmaxf(0.f, __fadd_rn(x.x, __fmaf_rn(dlt, __fadd_rn(x.x, x.y), -__fmul_rn(dld, x.y))));
        };
        bool use_w = !resid;
        float mine = 0.f;
        if (held) {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (c0 + i < c1) mine = __fadd_rn(mine, use_w ? q[i].x : mass_r(q[i]));
        } else {
            for (int c = c0; c < c1; ++c) mine = __fadd_rn(mine, use_w ? sub[c].x : mass_r(sub[c]));
        }
        if (resid && !(warp_sum(mine) > 0.f)) {
            // no residual mass (p = q up to rounding): draw from p.  Rare: the
            // chunk masses of p are formed here, one chunk at a time.
            use_w = true;
            mine = 0.f;
            const float2 l2 = make_float2(si.l_t, 0.f);
            for (int c = 0; c < nch; ++c) {
                float w = 0.f;
#pragma unroll
                for (int i = 0; i < kVecPerLane; ++i) {
                    const uint4 v = load_vec<DT, VEC>(rowt, (long long)c * CE + (long long)(i * 32 + lane) * EPV, P.V);
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        w = __fadd_rn(w, weight2l(make_float2(elem<DT>(v, e), -INFINITY), m2, chi2, clo2, l2).x);
                }
                w = warp_sum(w);
                if (lane == 0) sub[c].x = w;  // this warp alone reads request b's records
            }
            __syncwarp();
            __threadfence_block();
            if (held) {
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) q[i] = c0 + i < c1 ? sub[c0 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (int c = c0; c < c1; ++c) mine = __fadd_rn(mine, sub[c].x);
        }
        // two-float inclusive prefix over the lanes, then theta = u * Z
        FF incl{mine, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const FF t{__shfl_up_sync(0xFFFFFFFFu, incl.hi, o), __shfl_up_sync(0xFFFFFFFFu, incl.lo, o)};
            if (lane >= o) incl = ff_add(incl, t);
        }
        const FF Z{__shfl_sync(0xFFFFFFFFu, incl.hi, 31), __shfl_sync(0xFFFFFFFFu, incl.lo, 31)};
        const double theta = si.u * ((double)Z.hi + (double)Z.lo);
        const FF excl = ff_add(incl, FF{-mine, 0.f});
        float rem = (float)(theta - ((double)excl.hi + (double)excl.lo));  // mass left at this block
        const bool mine_crosses = rem >= 0.f && rem < mine;
        int my_c = INT_MAX, my_last = -1;
        float my_rem = 0.f;
        auto visit = [&](int c, const float4 &x) {
            const float v = use_w ? x.x : mass_r(x);
            if (v > 0.f) my_last = c;
            if (mine_crosses && my_c == INT_MAX) {
                if (v > rem) {
                    my_c = c;
                    my_rem = rem;
                }
                rem = __fsub_rn(rem, v);
            }
        };
        if (held) {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (c0 + i < c1) visit(c0 + i, q[i]);
        } else {
            for (int c = c0; c < c1; ++c) visit(c, sub[c]);
        }
        const int ch_found = warp_min_int(my_c);
        int ch;
        float th;  // mass left inside the chosen chunk
        if (ch_found != INT_MAX) {
            ch = ch_found;
            const int owner = __ffs(__ballot_sync(0xFFFFFFFFu, my_c == ch_found)) - 1;
            th = __shfl_sync(0xFFFFFFFFu, my_rem, owner);
        } else {
            // rounding left no crossing: the last chunk with positive mass
            int last = my_last;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xFFFFFFFFu, last, o));
            ch = last >= 0 ? last : nch - 1;
            th = INFINITY;
        }
        if (lane == 0) {
            s_ch = ch;
            s_th = th;
            s_two = resid && !use_w;
            s_dlt = dlt;
            s_dld = dld;
        }
    }
    __syncthreads();
    // the chosen chunk: thread t owns vectors t * kFindVecs .. t * kFindVecs + kFindVecs - 1
    const int ch = s_ch;
    const float th = s_th, dlt = s_dlt, dld = s_dld;  // th: mass left inside the chunk
    const bool two = s_two != 0;
    const float2 l2 = two ? make_float2(si.l_t, si.l_d) : make_float2(si.l_t, 0.f);
    const long long e0 = (long long)ch * CE + (long long)threadIdx.x * kFindVecs * EPV;
    uint4 vt[kFindVecs], vd[kFindVecs];
#pragma unroll
    for (int i = 0; i < kFindVecs; ++i) {
        vt[i] = load_vec<DT, VEC>(rowt, e0 + (long long)i * EPV, P.V);
        vd[i] = two ? load_vec<DT, VEC>(rowd, e0 + (long long)i * EPV, P.V) : neg_inf;
    }
    float vs[kFindVecs];
    float tot = 0.f;
    int last_pos = -1;
#pragma unroll
    for (int i = 0; i < kFindVecs; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const float w = draw_weight<DT>(
                weight2l(make_float2(elem<DT>(vt[i], e), elem<DT>(vd[i], e)), m2, chi2, clo2, l2), two, dlt, dld);
            acc = __fadd_rn(acc, w);
            if (w > 0.f && e0 + i * EPV + e < P.V) last_pos = (int)(e0 + i * EPV + e);
        }
        vs[i] = acc;
        tot = __fadd_rn(tot, acc);
    }
    float inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc = __fadd_rn(inc, u);
    }
    if (lane == 31) s_wt[warp] = inc;
    __syncthreads();
    float woff = 0.f;  // the mass of the warps before this one, added in warp order
    for (int j = 0; j < warp; ++j) woff = __fadd_rn(woff, s_wt[j]);
    const float lo = __fadd_rn(woff, __fsub_rn(inc, tot));
    int tok = INT_MAX;
    if (lo <= th && __fadd_rn(lo, tot) > th) {  // the crossing lane walks its elements in order
        float acc_lo = lo;
        bool done = false;
#pragma unroll
        for (int i = 0; i < kFindVecs; ++i) {
            if (!done && __fadd_rn(acc_lo, vs[i]) > th) {
                float ps = acc_lo;
                int lastp = -1;
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const float w = draw_weight<DT>(
                        weight2l(make_float2(elem<DT>(vt[i], e), elem<DT>(vd[i], e)), m2, chi2, clo2, l2), two,
                        dlt, dld);
                    ps = __fadd_rn(ps, w);
                    if (w > 0.f) lastp = (int)(e0 + i * EPV + e);
                    if (tok == INT_MAX && ps > th) tok = (int)(e0 + i * EPV + e);
                }
                if (tok == INT_MAX) tok = lastp;  // rounding inside the vector: its last positive element
                done = true;
            }
            if (!done) acc_lo = __fadd_rn(acc_lo, vs[i]);
        }
        if (tok < 0) tok = INT_MAX;
    }
    tok = warp_min_int(tok);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) last_pos = max(last_pos, __shfl_xor_sync(0xFFFFFFFFu, last_pos, o));
    if (lane == 0) {
        s_tok[warp] = tok;
        s_last[warp] = last_pos;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int found = INT_MAX, lp = -1;
        for (int j = 0; j < kFindWarps; ++j) {
            found = min(found, s_tok[j]);
            lp = max(lp, s_last[j]);
        }
        if (found == INT_MAX) found = lp >= 0 ? lp : (int)((long long)ch * CE);
        P.out_tokens[(size_t)b * (P.K + 1) + si.a] = found;
    }
}

// ------------------------------------------------------------------ schedule

__global__ void sv_schedule(const float *__restrict__ mp, float thr, int B, int K,
                            int32_t *__restrict__ out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    out[b] = schedule_threshold(mp + (size_t)b * K, K, thr);
}

// ------------------------------------------------------------------ draft confidence

// Rows of the draft-confidence pass: every draft row of every sampled request
// (a greedy request's draft distribution is a point mass).
__global__ void __launch_bounds__(kPrepThreads) sv_conf_rows(Params P) {
    __shared__ int warp_tot[kPrepThreads / 32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    pdl_trigger();
    for (int base = 0; base < P.B; base += kPrepThreads) {
        const int b = base + tid;
        int n = 0;
        float cval = 0.f;
        if (b < P.B) {
            const float T = P.temperature[b];
            if (isfinite(T) && T >= FLT_MIN) {
                n = P.K;
                cval = __fdiv_rn(kLog2EHi, T);
            }
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_tot[w] = incl;
        __syncthreads();
        int woff = 0, block_tot = 0;
        for (int i = 0; i < kPrepThreads / 32; ++i) {
            if (i < w) woff += warp_tot[i];
            block_tot += warp_tot[i];
        }
        const int off = carry_s + woff + incl - n;
        for (int r = 0; r < n; ++r) P.rows[off + r] = make_int4(b, P.K + 1 + r, 0, __float_as_int(cval));
        __syncthreads();
        if (tid == 0) carry_s += block_tot;
        __syncthreads();
    }
    if (tid == 0) *P.row_count = carry_s;
}

// max_v q(v) = 1 / sum_v 2^((z_v - m) log2(e)/T) of draft row (b, k), one warp
// per row from the statistics pass's partials; 1 for greedy requests.
__global__ void __launch_bounds__(kThreads) sv_conf_out(Params P, float *maxprob) {
    pdl_wait();  // partials come from sv_pass1
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= (long long)P.B * P.K) return;
    const int b = (int)(row / P.K), k = (int)(row - (long long)b * P.K);
    const float T = P.temperature[b];
    float out = 1.0f;
    if (isfinite(T) && T >= FLT_MIN) {
        const float4 rs = combine_row(P, b, P.K + 1 + k, false, __fdiv_rn(kLog2EHi, T), lane);
        out = __frcp_rn(rs.y);
    }
    if (lane == 0) maxprob[row] = out;
}

// ------------------------------------------------------------------ tree verification (greedy)

// Rows of a greedy tree verification: every node row of every request (the
// target logits [B, N, V] sit where the target rows 0..K of a K = N - 1 call
// would).
__global__ void sv_tree_rows(Params P) {
    pdl_trigger();
    const int n = P.K + 1;
    const long long total = (long long)P.B * n;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x)
        P.rows[i] = make_int4((int)(i / n), (int)(i % n), 1, 0);
    if (blockIdx.x == 0 && threadIdx.x == 0) *P.row_count = (int)total;
}

// A node whose parent is not an earlier node belongs to no path; such a tree
// raises SPEC_DEV_BAD_TREE.
__device__ __forceinline__ void flag_bad_tree(const Params &P, int N, const int *s_par) {
    bool bad = false;
    for (int c = 1; c < N; ++c) bad |= s_par[c] < 0 || s_par[c] >= c;
    if (bad && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_BAD_TREE);
}

// One thread: the greedy walk of request b from the argmax of every node row.
__device__ void greedy_tree_walk(const Params &P, int b, int N, const int *s_amax,
                                 const int *s_par, const int *s_tok, int32_t *out_nodes) {
    int32_t *out = P.out_tokens + (size_t)b * N;
    int32_t *nodes = out_nodes + (size_t)b * N;
    int cur = 0, depth = 0;
    for (;;) {
        const int t = s_amax[cur];
        int next = -1;
        for (int c = cur + 1; c < N; ++c)
            if (s_par[c] == cur && s_tok[c] == t) {
                next = c;
                break;
            }
        out[depth] = t;
        if (next < 0) break;
        nodes[depth] = next;
        cur = next;
        ++depth;
    }
    for (int i = depth + 1; i < N; ++i) out[i] = -1;
    for (int i = depth; i < N; ++i) nodes[i] = -1;
    P.accept_len[b] = depth;
    flag_bad_tree(P, N, s_par);
}

// Per request: the argmax of every node row from the statistics pass's
// partials, then the walk from the root -- t = argmax of the current node, the
// next node is the lowest-index child carrying t, else t is emitted.  A node
// whose parent is not an earlier node belongs to no path (SPEC_DEV_BAD_TREE).
__global__ void __launch_bounds__(kThreads) sv_tree_decide(Params P, const int32_t *parent,
                                                          const int32_t *token,
                                                          int32_t *out_nodes) {
    __shared__ int s_amax[SPEC_MAX_TREE];
    __shared__ int s_par[SPEC_MAX_TREE], s_tok[SPEC_MAX_TREE];
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = P.K + 1;
    for (int i = tid; i < N; i += kThreads) {
        s_par[i] = parent[(size_t)b * N + i];
        s_tok[i] = token[(size_t)b * N + i];
    }
    pdl_wait();  // partials come from sv_pass1
    pdl_trigger();
    for (int n = warp; n < N; n += kWarps) {
        const float4 rs = combine_row(P, b, n, true, 0.f, lane);
        if (lane == 0) s_amax[n] = __float_as_int(rs.z);
    }
    __syncthreads();
    if (tid == 0) greedy_tree_walk(P, b, N, s_amax, s_par, s_tok, out_nodes);
}

// ------------------------------------------------------------------ tree verification (sampled)

// Rows of a tree verification with sampled requests: every node row of the
// target (slots 0..N-1) and, for sampled requests, the draft rows 0..N-2
// (slots N..2N-2; draft row n is the distribution node n's children were drawn
// from, and the last node has no children).  Request-major, one CTA.
__global__ void __launch_bounds__(kPrepThreads) sv_tree_rows_s(Params P) {
    __shared__ int warp_tot[kPrepThreads / 32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int N = P.K + 1;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    pdl_trigger();
    for (int base = 0; base < P.B; base += kPrepThreads) {
        const int b = base + tid;
        int n = 0, greedy = 1;
        float cval = 0.f;
        if (b < P.B) {
            const float T = P.temperature[b];
            greedy = !(isfinite(T) && T >= FLT_MIN);
            if (!greedy) cval = __fdiv_rn(kLog2EHi, T);
            n = greedy ? N : 2 * N - 1;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_tot[w] = incl;
        __syncthreads();
        int woff = 0, block_tot = 0;
        for (int i = 0; i < kPrepThreads / 32; ++i) {
            if (i < w) woff += warp_tot[i];
            block_tot += warp_tot[i];
        }
        const int off = carry_s + woff + incl - n;
        for (int r = 0; r < n; ++r)
            P.rows[off + r] = make_int4(b, r, greedy, __float_as_int(cval));
        __syncthreads();
        if (tid == 0) carry_s += block_tot;
        __syncthreads();
    }
    if (tid == 0) *P.row_count = carry_s;
}

constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeStep = 256;     // elements a warp covers per step: 8 per lane
constexpr int kTreeGroups = 256;   // recorded masses per warp (groups of steps)
constexpr float kTreeBias = 2.0f;  // every summed weight is at most ~1
constexpr int kTreeStageMax = 176 * 1024;  // dynamic shared memory for a staged slice (two rows)

// The weight 2^(z c + base) of one element, base = l - m c for a row with
// max m and log2(1/S) = l: one FMA per element.  The rounding of base scales
// every weight of the row alike, which the exact normalisers (the sums of the
// same weights) remove.  wpair is the twin for an element pair (the same
// operations, so the same values).
__device__ __forceinline__ float weight1b(float z, float c, float base) {
    return ex2(__fmaf_rn(z, c, base));
}
__device__ __forceinline__ float2 wpair(float2 z, float2 c2, float2 base2) {
    const float2 t = fma2(z, c2, base2);
    return make_float2(ex2(t.x), ex2(t.y));
}
__device__ __forceinline__ float row_base(float m, float c, float l) {
    return __fmaf_rn(-m, c, l);
}

// Residual after j rejected siblings, in closed form.  With p, q the target
// and draft distributions, r_1 = max(0, p - q) and r_(j+1) = max(0, r_j / Z_j
// - q) give r_j = c_j max(0, p - t_j q) for a scale c_j and the threshold
// t_1 = 1, t_(j+1) = t_j + sum_v max(0, p - t_j q): the scale cancels in the
// acceptance test and the inverse CDF, so only the threshold is carried.  In
// the weights a, b (p = a / A, q = b / B with A, B their exact sums) the
// residual is proportional to max(0, a - s b), s = t A / B, and
// s_1 = A / B, s_(j+1) = s_j + S_j / B with S_j = sum_v max(0, a - s_j b).
// s = 0 stands for the weights p themselves (a restart after zero mass).
__device__ __forceinline__ float resid_weight(float a, float b, float s) {
    return fmaxf(__fmaf_rn(-s, b, a), 0.f);
}

// Elements [e0, e0 + 8) of a row as 4 pairs (-inf past V).
template <int DT, bool VEC> struct Eight {
    uint4 v0, v1;
    __device__ __forceinline__ void load(const char *row, long long e0, int V) {
        v0 = load_vec<DT, VEC>(row, e0, V);
        if (DT == kF32) v1 = load_vec<DT, VEC>(row, e0 + 4, V);
    }
    // the same elements from a staged copy in shared memory (stage = the
    // element at index 0 of the copy, i0 = e0's index there; V a multiple of
    // the 16-byte vector, so each vector lies wholly before or past V)
    __device__ __forceinline__ void load_staged(const char *stage, int i0, long long e0, int V) {
        const uint32_t ni = Fmt<DT>::kNegInfWord;
        const uint4 neg = make_uint4(ni, ni, ni, ni);
        v0 = e0 < V ? *reinterpret_cast<const uint4 *>(stage + (size_t)i0 * Fmt<DT>::kESZ) : neg;
        if (DT == kF32)
            v1 = e0 + 4 < V ? *reinterpret_cast<const uint4 *>(stage + (size_t)(i0 + 4) * Fmt<DT>::kESZ)
                            : neg;
    }
    __device__ __forceinline__ float2 pair(int i) const {
        if (DT == kBF16) return make_float2(elem<DT>(v0, 2 * i), elem<DT>(v0, 2 * i + 1));
        return i < 2 ? make_float2(elem<DT>(v0, 2 * i), elem<DT>(v0, 2 * i + 1))
                     : make_float2(elem<DT>(v1, 2 * i - 4), elem<DT>(v1, 2 * i - 3));
    }
};

// Per-node constants of the sampled walk.
struct TreeNodeC {
    float2 bt, bd, c2;  // weight bases of the target and draft rows (row_base), log2(e)/T
    float s;                          // residual threshold (0: the weights p)
};

// Weights a pass sums: the target weights a; the parts of the first residual
// (sum a, sum b, sum over a > b of (a - b), sum over a > b of b); the residual
// max(0, a - s b).
enum { kTreeModeP = 0, kTreeModeFirst = 1, kTreeModeThr = 2 };

// The 8 weights of a lane in a pass of mode P or Thr.
template <int DT, bool VEC>
__device__ __forceinline__ void tree_weights8(const Eight<DT, VEC> &zt, const Eight<DT, VEC> &zd,
                                              const TreeNodeC &nc, int mode, float w[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = wpair(zt.pair(i), nc.c2, nc.bt);
        if (mode == kTreeModeP) {
            w[2 * i] = a.x;
            w[2 * i + 1] = a.y;
        } else {
            const float2 bq = wpair(zd.pair(i), nc.c2, nc.bd);
            w[2 * i] = resid_weight(a.x, bq.x, nc.s);
            w[2 * i + 1] = resid_weight(a.y, bq.y, nc.s);
        }
    }
}

// The CTAs of a cluster share one request: CTA `rank` of `cs` covers a
// contiguous slice of the steps of kTreeStep elements, and its warp w the
// steps [s0, s1) of that slice; recorded masses cover groups of gsz
// consecutive steps.
struct TreeSplit {
    int c0, s0, s1, gsz;
    __device__ __forceinline__ TreeSplit(int V, int rank, int cs, int w) {
        const int nsteps = (V + kTreeStep - 1) / kTreeStep;
        const int spc = (nsteps + cs - 1) / cs;
        c0 = min(nsteps, rank * spc);
        const int c1 = min(nsteps, c0 + spc);
        const int spw = (c1 - c0 + kTreeWarps - 1) / kTreeWarps;
        s0 = min(c1, c0 + w * spw);
        s1 = min(c1, s0 + spw);
        gsz = max(1, (spw + kTreeGroups - 1) / kTreeGroups);
    }
};

// Cluster primitives: this CTA's rank and the cluster's size, a barrier of all
// threads of the cluster (release / acquire), and a double read from the
// shared memory of CTA `rank` at the address of `local` in this CTA.
__device__ __forceinline__ int cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}
__device__ __forceinline__ int cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return (int)r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ double ld_cluster_f64(const double *local, int rank) {
    uint32_t ra;
    double v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(ra) : "memory");
    return v;
}

// Warp 0 of a CTA: the sums red[w][i] (i < n) of its warps into slot[i], added
// by a fixed shuffle tree.
__device__ __forceinline__ void warp_sums_to_slot(const double (*red)[4], double *slot, int n,
                                                  int lane) {
    for (int i = 0; i < n; ++i) {
        const double v = warp_sum_d(lane < kTreeWarps ? red[lane][i] : 0.0);
        if (lane == 0) slot[i] = v;
    }
}

// Warp 0: the cluster totals of slot[0..n) (n <= 4, cs <= 8).  Lane 4 r + i
// reads slot[i] of CTA r; a fixed shuffle tree adds over r, so every CTA
// obtains the same bits.  Every lane receives tot[0..n).
__device__ __forceinline__ void cluster_totals(const double *slot, int n, int cs, int lane,
                                               double tot[4]) {
    const int r = lane >> 2, i = lane & 3;
    double v = (r < cs && i < n) ? ld_cluster_f64(&slot[i], r) : 0.0;
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) tot[k] = __shfl_sync(0xFFFFFFFFu, v, k);
}

// Warp 0: the first of n masses (lane j holds m, 0 past n) whose inclusive
// prefix from base exceeds thr, and the mass before it; rounding that leaves
// no crossing takes the last positive mass.  Returns -1 when all are 0.
__device__ __forceinline__ int crossing_lane(double m, double base, double thr, int lane,
                                             double &before) {
    double incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    const unsigned cross = __ballot_sync(0xFFFFFFFFu, m > 0.0 && base + incl > thr);
    const unsigned has = __ballot_sync(0xFFFFFFFFu, m > 0.0);
    if (!has) return -1;
    const int j = cross ? __ffs(cross) - 1 : 31 - __clz(has);
    before = base + __shfl_sync(0xFFFFFFFFu, incl - m, j);
    return j;
}

// One pass of the CTA over its slice of the vocabulary.  Warp w covers its contiguous steps,
// lane l the 8 elements at 8 l of each step, kU steps' loads in flight.  Writes
// the warp's sums (as doubles) to red[w]; with `record`, also the mass of each
// group of steps to mass[w * kTreeGroups + g] and the warp's total as their sum.
// Mode First with `record` (the first residual's threshold is not known yet):
// red[w] = {sum a, sum b (exact), sum over a > b of (a - b), of b}, the last
// two also per group, in mass[] and mass2[].
template <int DT, bool VEC>
__device__ void tree_pass(const char *rowt, const char *rowd, const char *stt, const char *std_,
                          int V, int rank, int cs, const TreeNodeC &nc, int mode, bool record,
                          double (*red)[4], float *mass, float *mass2, int warp, int lane) {
    constexpr int kU = DT == kBF16 ? 2 : 1;  // steps per batch; two batches in flight
    const TreeSplit sp(V, rank, cs, warp);
    BiasAcc2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i].init(kTreeBias);
    float gs = 0.f, gs2 = 0.f;  // this lane's parts of the current group
    double mw = 0.0, mw2 = 0.0;  // the warp's recorded totals (lane 0)
    // close the group of step st (the last of its group or of the warp's steps)
    auto close_group = [&](int st, bool two) {
        const int k = st - sp.s0;
        if ((k + 1) % sp.gsz == 0 || st + 1 == sp.s1) {
            const float gm = warp_sum(gs);
            const float gm2 = two ? warp_sum(gs2) : 0.f;
            if (lane == 0) {
                mass[warp * kTreeGroups + k / sp.gsz] = gm;
                mw += (double)gm;
                if (two) {
                    mass2[warp * kTreeGroups + k / sp.gsz] = gm2;
                    mw2 += (double)gm2;
                }
            }
            gs = 0.f;
            gs2 = 0.f;
        }
    };
    auto load = [&](Eight<DT, VEC> (&zt)[kU], Eight<DT, VEC> (&zd)[kU], int st0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const long long e0 = (long long)(st0 + u) * kTreeStep + lane * 8;
            if (st0 + u < sp.s1) {
                if (stt) {  // staged slice of this CTA
                    const int i0 = (st0 + u - sp.c0) * kTreeStep + lane * 8;
                    zt[u].load_staged(stt, i0, e0, V);
                    if (mode != kTreeModeP) zd[u].load_staged(std_, i0, e0, V);
                } else {
                    zt[u].load(rowt, e0, V);
                    if (mode != kTreeModeP) zd[u].load(rowd, e0, V);
                }
            }
        }
    };
    auto consume = [&](const Eight<DT, VEC> (&zt)[kU], const Eight<DT, VEC> (&zd)[kU], int st0) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (st0 + u >= sp.s1) break;
            if (mode == kTreeModeFirst) {
                float ld = 0.f, lb = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 a = wpair(zt[u].pair(i), nc.c2, nc.bt);
                    const float2 bq = wpair(zd[u].pair(i), nc.c2, nc.bd);
                    acc[0].add(a);
                    acc[1].add(bq);
                    const bool gx = a.x > bq.x, gy = a.y > bq.y;
                    const float2 dd = make_float2(gx ? __fsub_rn(a.x, bq.x) : 0.f,
                                                  gy ? __fsub_rn(a.y, bq.y) : 0.f);
                    const float2 bb = make_float2(gx ? bq.x : 0.f, gy ? bq.y : 0.f);
                    if (record) {
                        ld = __fadd_rn(ld, __fadd_rn(dd.x, dd.y));
                        lb = __fadd_rn(lb, __fadd_rn(bb.x, bb.y));
                    } else {
                        acc[2].add(dd);
                        acc[3].add(bb);
                    }
                }
                if (record) {
                    gs = __fadd_rn(gs, ld);
                    gs2 = __fadd_rn(gs2, lb);
                    close_group(st0 + u, true);
                }
            } else {
                float w[8];
                tree_weights8<DT, VEC>(zt[u], zd[u], nc, mode, w);
                if (record) {
                    float ls = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) ls = __fadd_rn(ls, w[i]);
                    gs = __fadd_rn(gs, ls);
                    close_group(st0 + u, false);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[0].add(make_float2(w[2 * i], w[2 * i + 1]));
                }
            }
        }
    };
    // batch A holds steps [st0, st0 + kU), batch B the next kU: one is loading
    // while the other is consumed
    Eight<DT, VEC> ta[kU], da[kU], tb[kU], db[kU];
    load(ta, da, sp.s0);
    for (int st0 = sp.s0; st0 < sp.s1; st0 += 2 * kU) {
        load(tb, db, st0 + kU);
        consume(ta, da, st0);
        load(ta, da, st0 + 2 * kU);
        consume(tb, db, st0 + kU);
    }
    if (record && mode == kTreeModeFirst) {
        const FF ta = warp_sum_ff(acc[0].total()), tb = warp_sum_ff(acc[1].total());
        if (lane == 0) {
            red[warp][0] = ff_to_double(ta);
            red[warp][1] = ff_to_double(tb);
            red[warp][2] = mw;
            red[warp][3] = mw2;
        }
        return;
    }
    if (record) {
        if (lane == 0) red[warp][0] = mw;
        return;
    }
    const int nsum = mode == kTreeModeFirst ? 4 : 1;
    for (int i = 0; i < nsum; ++i) {
        const FF t = warp_sum_ff(acc[i].total());
        if (lane == 0) red[warp][i] = ff_to_double(t);
    }
}

// The emitted token, by one warp: the inverse CDF of the weights of the last
// recording pass at thr, inside warp W's steps (base = the mass of the warps
// before W): the group whose prefix crosses thr, then the step, then the
// element.  Rounding that leaves the crossing outside takes the last positive
// weight met.
template <int DT, bool VEC>
__device__ int tree_find(const char *rowt, const char *rowd, const char *stt, const char *std_,
                         int V, int rank, int cs, const TreeNodeC &nc, int mode, const float *mass,
                         int W, double base, double thr, int lane) {
    const TreeSplit sp(V, rank, cs, W);
    const int ng = (sp.s1 - sp.s0 + sp.gsz - 1) / sp.gsz;
    constexpr int kPer = kTreeGroups / 32;  // lane l holds groups [kPer l, kPer (l + 1))
    static_assert(kPer == 8, "the lane sum below adds 8 group masses");
    float gm[kPer];
    double t8[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int g = lane * kPer + i;
        gm[i] = g < ng ? mass[W * kTreeGroups + g] : 0.f;
        t8[i] = (double)gm[i];
    }
    const double ls = ((t8[0] + t8[1]) + (t8[2] + t8[3])) + ((t8[4] + t8[5]) + (t8[6] + t8[7]));
    double incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    const unsigned cross = __ballot_sync(0xFFFFFFFFu, base + incl > thr && ls > 0.0);
    const unsigned has = __ballot_sync(0xFFFFFFFFu, ls > 0.0);
    if (!has) return -1;
    // the crossing lane, else (rounding) the last lane with mass
    const int src = cross ? __ffs(cross) - 1 : 31 - __clz(has);
    int g = -1;
    double gbase = 0.0;
    if (lane == src) {
        double c = base + incl - ls;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (gm[i] > 0.f && (g < 0 || c <= thr)) {
                g = lane * kPer + i;
                gbase = c;
            }
            c += (double)gm[i];
        }
    }
    g = __shfl_sync(0xFFFFFFFFu, g, src);
    gbase = __shfl_sync(0xFFFFFFFFu, gbase, src);
    // the steps of group g, in order
    const int st_a = sp.s0 + g * sp.gsz, st_b = min(sp.s1, st_a + sp.gsz);
    double b0 = gbase;
    int last_pos = -1;
    for (int st = st_a; st < st_b; ++st) {
        const long long e0 = (long long)st * kTreeStep + lane * 8;
        Eight<DT, VEC> zt, zd;
        if (stt) {
            const int i0 = (st - sp.c0) * kTreeStep + lane * 8;
            zt.load_staged(stt, i0, e0, V);
            if (mode != kTreeModeP) zd.load_staged(std_, i0, e0, V);
        } else {
            zt.load(rowt, e0, V);
            if (mode != kTreeModeP) zd.load(rowd, e0, V);
        }
        float w[8];
        tree_weights8<DT, VEC>(zt, zd, nc, mode, w);
        int lp = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (w[i] > 0.f) lp = (int)e0 + i;
        const double s8 = (((double)w[0] + (double)w[1]) + ((double)w[2] + (double)w[3])) +
                          (((double)w[4] + (double)w[5]) + ((double)w[6] + (double)w[7]));
        double in8 = s8;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double v = __shfl_up_sync(0xFFFFFFFFu, in8, o);
            if (lane >= o) in8 += v;
        }
        const unsigned cr = __ballot_sync(0xFFFFFFFFu, b0 + in8 > thr && s8 > 0.0);
        const int lp_max = (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)(lp + 1)) - 1;
        if (cr) {
            const int L = __ffs(cr) - 1;
            int tok = -1;
            if (lane == L) {
                double c = b0 + in8 - s8;
                for (int i = 0; i < 8 && tok < 0; ++i) {
                    c += (double)w[i];
                    if (w[i] > 0.f && c > thr) tok = (int)e0 + i;
                }
                if (tok < 0) tok = lp;
            }
            return __shfl_sync(0xFFFFFFFFu, tok, L);
        }
        if (lp_max >= 0) last_pos = lp_max;
        b0 += __shfl_sync(0xFFFFFFFFu, in8, 31);
    }
    return last_pos;
}

// Sampled verification of candidate trees by a cluster of CTAs per request
// (greedy requests take the greedy walk).  At node u the first child is
// checked with the linear acceptance test; after j rejections the residual is
// max(0, a - s_j b) (see resid_weight), and a rejection followed by another
// candidate costs one pass over the vocabulary for the residual's mass S_j,
// against which the next sibling is checked: accept iff
// u_acc * b(x) * S_j < B * max(0, a(x) - s_j b(x)).  When no child is accepted
// a recording pass over the current weights and an inverse CDF give the
// emitted token.  Candidate node c takes the acceptance uniform of position
// c - 1, node u's emitted token the sampling uniform of position u.
// distinct: the siblings were drawn without replacement from q_u, so the
// draft law of the sibling after j rejections is q without the rejected
// tokens, divided by their remaining mass 1 - Q_j.  The residual keeps the
// same closed form with the threshold step divided by that mass, and the test
// is scaled by it: with R_j = B - sum of b over the rejected tokens (= B (1 -
// Q_j)), accept iff u_acc * b(x) * S_j < R_j * max(0, a(x) - s_j b(x)), and
// s_(j+1) = s_j + S_j / R_j (s_j = A / R_(j-1) after a restart from p).  A
// sibling repeating a rejected token, or met when R_j <= 0, is no candidate.
// Each CTA of the cluster passes over its slice of the vocabulary; the sums
// are exchanged through distributed shared memory and added by the same fixed
// shuffle tree in every CTA, so all CTAs take the same decisions and meet the
// same cluster barriers.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kTreeThreads, 1) sv_tree_walk(Params P, const int32_t *parent,
                                                               const int32_t *token,
                                                               int32_t *out_nodes,
                                                               int stage_row_bytes, int diag,
                                                               int distinct) {
    // stage_row_bytes > 0: this CTA's slice of a node's target and draft rows is
    // copied into dynamic shared memory at the node's first rejection, and the
    // node's later passes read it there.  diag: before each staging wait, every
    // warp first waits on a barrier nothing completes, gives up after
    // kDiagWaitNs and reports SPEC_DEV_TIMEOUT as on a real timeout (the real
    // wait follows, so the results are unchanged).
    extern __shared__ __align__(128) unsigned char s_stage[];
    __shared__ uint64_t s_tbar[kTreeWarps], s_never;
    __shared__ int s_par[SPEC_MAX_TREE], s_tok[SPEC_MAX_TREE], s_amax[SPEC_MAX_TREE];
    __shared__ float s_m[2 * SPEC_MAX_TREE], s_S[2 * SPEC_MAX_TREE];
    __shared__ float s_u[SPEC_MAX_TREE], s_g[SPEC_MAX_TREE], s_gd[SPEC_MAX_TREE];
    __shared__ double s_us[SPEC_MAX_TREE];
    __shared__ float s_mass[kTreeWarps * kTreeGroups];
    __shared__ float s_mass2[kTreeWarps * kTreeGroups];  // a merged first pass: sum of b per group
    __shared__ double s_red[kTreeWarps][4];
    __shared__ double s_slot[2][4];   // this CTA's sums, read by the cluster (two buffers)
    __shared__ double s_sum;          // S_j of the current residual
    __shared__ double s_SA, s_SB;     // exact sums of a and b at the node
    __shared__ double s_iSB;          // 1 / s_SB
    __shared__ int s_cand[SPEC_MAX_TREE], s_ncand;  // the current node's candidates, in order
    __shared__ double s_base, s_thr;
    __shared__ float s_s;
    __shared__ int s_acc, s_R, s_W, s_emit, s_again;
    __shared__ int s_nostage;  // a staging wait ran out: no more staging in this request
    __shared__ double s_brej;  // distinct: sum of b over the rejected siblings' tokens at the node
    __shared__ int s_rejtok[SPEC_MAX_TREE], s_nrej;  // distinct: those tokens
    constexpr int ESZ = Fmt<DT>::kESZ;
    const int cs = cluster_size(), rank = cluster_rank();
    const int b = blockIdx.x / cs, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = P.K + 1, K = P.K, V = P.V;
    const float T = P.temperature[b];
    const bool greedy = !(isfinite(T) && T >= FLT_MIN);
    // inputs only (nothing from the statistics pass): tree, uniforms, candidate logits
    for (int i = tid; i < N; i += kTreeThreads) {
        const int pa = parent[(size_t)b * N + i], x = token[(size_t)b * N + i];
        s_par[i] = pa;
        s_tok[i] = x;
        if (!greedy) {
            s_us[i] = uniform_sample(P.seed, (uint32_t)b, (uint32_t)i);
            if (i > 0) {
                s_u[i] = uniform_accept_f(P.seed, (uint32_t)b, (uint32_t)(i - 1));
                const bool ok = pa >= 0 && pa < i && x >= 0 && x < V;
                s_g[i] = ok ? load_logit(row_ptr(P, b, pa, ESZ), DT, x) : 0.f;
                s_gd[i] = ok ? load_logit(row_ptr(P, b, K + 1 + pa, ESZ), DT, x) : 0.f;
            }
        }
    }
    float c = 0.f, chi = 0.f, clo = 0.f;
    if (!greedy) temp_coeffs(T, c, chi, clo);
    if (lane == 0) mbar_init(&s_tbar[warp], 1);
    if (tid == 0) {
        mbar_init(&s_never, 1);
        s_nostage = 0;
    }
    fence_mbar_init();
    pdl_wait();  // partials come from sv_pass1
    pdl_trigger();
    const int nrows = greedy ? N : 2 * N - 1;
    for (int r = warp; r < nrows; r += kTreeWarps) {
        const float4 rs = combine_row(P, b, r, greedy, c, lane);
        if (lane == 0) {
            s_m[r] = rs.x;
            s_S[r] = rs.y;
            if (r < N) s_amax[r] = __float_as_int(rs.z);
        }
    }
    __syncthreads();
    if (greedy) {  // no cluster exchange: rank 0 walks, the others leave
        if (tid == 0 && rank == 0) greedy_tree_walk(P, b, N, s_amax, s_par, s_tok, out_nodes);
        return;
    }
    int32_t *out = P.out_tokens + (size_t)b * N;
    int32_t *nodes = out_nodes + (size_t)b * N;
    if (tid == 0 && rank == 0) flag_bad_tree(P, N, s_par);
    int par = 0;  // slot buffer of the next exchange
    uint32_t stagings = 0;  // copies into the staging buffer so far (phase of s_tbar)
    int cur = 0, depth = 0;
    for (;;) {
        const char *rowt = row_ptr(P, b, cur, ESZ);
        const bool inner = cur < N - 1;  // only such a node can have children (and a draft row)
        const char *rowd = inner ? row_ptr(P, b, K + 1 + cur, ESZ) : rowt;
        TreeNodeC nc;
        nc.c2 = make_float2(c, c);
        const float mt = s_m[cur], St = s_S[cur];
        const float md = inner ? s_m[K + 1 + cur] : 0.f, Sd = inner ? s_S[K + 1 + cur] : 1.f;
        const float lt = -log2f(St), ld = -log2f(Sd);
        const float bt = row_base(mt, c, lt), bd = row_base(md, c, ld);
        nc.bt = make_float2(bt, bt);
        nc.bd = make_float2(bd, bd);
        nc.s = 0.f;
        bool staged = false;  // this node's slice is in shared memory (this warp's steps)
        // the only candidate left was the first and it was rejected: the
        // recording pass also forms the exact sums (one pass instead of two)
        bool first_rec = false;
        if (warp == 0) {  // the children of cur with a token in [0, V), in index order
            int n = 0;
            for (int base = cur + 1; base < N; base += 32) {
                const int ch = base + lane;
                const bool ok = ch < N && s_par[ch] == cur && s_tok[ch] >= 0 && s_tok[ch] < V;
                const unsigned m = __ballot_sync(0xFFFFFFFFu, ok);
                if (ok) s_cand[n + __popc(m & ((1u << lane) - 1u))] = ch;
                n += __popc(m);
            }
            if (lane == 0) s_ncand = n;
        }
        if (tid == 0) {
            s_brej = 0.0;
            s_nrej = 0;
        }
        __syncthreads();
        const int ncand = s_ncand;
        int J = 0, next = -1;
        for (int k = 0; k < ncand; ++k) {
            const int ch = s_cand[k];
            if (tid == 0) {
                const float u = s_u[ch], g = s_g[ch], gd = s_gd[ch];
                int acc;  // 1 accepted, 0 rejected, -1 no candidate
                bool skip = false;
                if (distinct && J > 0) {  // a draw without replacement could not give it
                    const int x = s_tok[ch];
                    for (int i = 0; i < s_nrej; ++i) skip |= s_rejtok[i] == x;
                    skip |= !(s_SB - s_brej > 0.0);
                }
                if (skip) {
                    acc = -1;
                } else if (J == 0) {
                    acc = accept_position(u, g, mt, St, gd, md, Sd, chi, clo);
                } else {
                    const float a = weight1b(g, c, bt), bq = weight1b(gd, c, bd);
                    const float w = nc.s > 0.f ? resid_weight(a, bq, nc.s) : a;
                    acc = (double)u * (double)bq * s_sum < (double)w * (distinct ? s_SB - s_brej : s_SB);
                }
                s_acc = acc;
            }
            __syncthreads();
            const int decision = s_acc;
            if (decision < 0) {
                __syncthreads();  // s_acc is rewritten for the next candidate
                continue;
            }
            if (decision) {
                next = ch;
                break;
            }
            ++J;
            const bool more = k + 1 < ncand;  // another candidate follows: the residual's mass is needed
            if (J > 1) {  // the threshold after this rejection
                if (tid == 0) {
                    if (!distinct) {
                        s_s = nc.s > 0.f ? (float)((double)nc.s + s_sum * s_iSB) : (float)(s_SA * s_iSB);
                    } else {  // the remaining draft mass before this rejection
                        const double R = s_SB - s_brej;
                        s_s = nc.s > 0.f ? (float)((double)nc.s + s_sum / R) : (float)(s_SA / R);
                    }
                }
                __syncthreads();
                nc.s = s_s;
            }
            if (distinct && tid == 0) {  // this sibling's token leaves the draft law
                s_rejtok[s_nrej++] = s_tok[ch];
                s_brej += (double)weight1b(s_gd[ch], c, bd);
            }
            if (J > 1 && !more) break;  // the recording pass below needs no mass
            if (J == 1 && stage_row_bytes > 0 && !s_nostage) {  // every warp copies its own steps, then waits
                const TreeSplit sp(V, rank, cs, warp);
                fence_proxy_async();  // earlier reads of the buffer come first
                __syncwarp();
                if (lane == 0) {
                    const long long ea = (long long)sp.s0 * kTreeStep;
                    const long long eb = min((long long)sp.s1 * kTreeStep, (long long)V);
                    const uint32_t bytes = eb > ea ? (uint32_t)((eb - ea) * ESZ) : 0u;
                    unsigned char *dt = s_stage + (size_t)(sp.s0 - sp.c0) * kTreeStep * ESZ;
                    mbar_expect_tx(&s_tbar[warp], 2u * bytes);
                    if (bytes) {
                        bulk_g2s(dt, rowt + ea * ESZ, bytes, &s_tbar[warp]);
                        bulk_g2s(dt + stage_row_bytes, rowd + ea * ESZ, bytes, &s_tbar[warp]);
                    }
                }
                __syncwarp();
                if (diag && !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&s_never, 0u, kDiagWaitNs)) &&
                    lane == 0 && P.dev_status)
                    atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
                const bool ok = mbar_wait_bounded(&s_tbar[warp], stagings & 1u, kWaitLimitNs);
                staged = true;
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    // give up on staging: report, let this warp's copies land
                    // (bounded), read global memory from here on (the barrier's
                    // phase is no longer known, so the request stages no more)
                    if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
                    mbar_wait_bounded(&s_tbar[warp], stagings & 1u, kWaitLimitNs);
                    if (lane == 0) s_nostage = 1;
                    staged = false;
                }
                ++stagings;
            }
            if (J == 1 && !more) {
                first_rec = true;
                break;
            }
            const char *stt = staged ? (const char *)s_stage : nullptr;
            const char *std_ = staged ? (const char *)s_stage + stage_row_bytes : nullptr;
            const int mode = J == 1 ? kTreeModeFirst : kTreeModeThr;
            tree_pass<DT, VEC>(rowt, rowd, stt, std_, V, rank, cs, nc, mode, false, s_red, s_mass, s_mass2,
                               warp, lane);
            __syncthreads();
            const int nsum = mode == kTreeModeFirst ? 4 : 1;
            if (warp == 0) warp_sums_to_slot(s_red, s_slot[par], nsum, lane);
            cluster_sync_all();
            double tot[4];
            if (warp == 0) cluster_totals(s_slot[par], nsum, cs, lane, tot);
            if (tid == 0) {
                double S;
                if (mode == kTreeModeFirst) {
                    s_SA = tot[0];
                    s_SB = tot[1];
                    s_iSB = 1.0 / tot[1];
                    const float s1 = (float)(tot[0] * s_iSB);
                    // sum over a > b of (a - s_1 b): the residual max(0, a - s_1 b)
                    // summed over a > b instead of a > s_1 b.  The two supports
                    // differ only where a lies between b and s_1 b; with
                    // |s_1 - 1| ~ 1e-6 (both weight sets are normalised to ~1)
                    // the mass differs by at most |s_1 - 1| times the draft mass
                    // of those near ties, far below the acceptance window.
                    S = tot[2] + (1.0 - (double)s1) * tot[3];
                    s_s = s1;
                } else {
                    S = tot[0];
                    s_s = nc.s;
                }
                if (!(S > 0.0)) {  // no residual mass: the weights restart from p
                    s_s = 0.f;
                    S = s_SA;
                }
                s_sum = S;
            }
            par ^= 1;
            __syncthreads();
            nc.s = s_s;
            if (!more) break;
        }
        if (next >= 0) {
            if (tid == 0 && rank == 0) {
                out[depth] = s_tok[next];
                nodes[depth] = next;
            }
            cur = next;
            ++depth;
            __syncthreads();  // s_acc and the sums are rewritten at the next node
            continue;
        }
        // no child accepted: the emitted token from the current weights (a warp
        // whose staging gave up reads global memory; tree_find below reads
        // another warp's steps, so it takes the staged copy only if no warp gave up)
        const char *stt = staged ? (const char *)s_stage : nullptr;
        const char *std_ = staged ? (const char *)s_stage + stage_row_bytes : nullptr;
        for (;;) {
            const int mode = first_rec ? kTreeModeFirst : nc.s > 0.f ? kTreeModeThr : kTreeModeP;
            tree_pass<DT, VEC>(rowt, rowd, stt, std_, V, rank, cs, nc, mode, true, s_red, s_mass, s_mass2,
                               warp, lane);
            __syncthreads();
            if (warp == 0) warp_sums_to_slot(s_red, s_slot[par], first_rec ? 4 : 1, lane);
            cluster_sync_all();
            double k1 = 0.0;  // merged first pass: 1 - s_1
            if (first_rec) {
                // s_1 = A / B from the exact sums, then the residual max(0, a - s_1 b)
                // of each group and warp as D + (1 - s_1) Bm over a > b (the two
                // supports differ only at near ties, as for the mass S_1 above)
                double tot[4];
                if (warp == 0) cluster_totals(s_slot[par], 4, cs, lane, tot);
                if (tid == 0) {
                    s_SA = tot[0];
                    s_SB = tot[1];
                    s_iSB = 1.0 / tot[1];
                    s_s = (float)(tot[0] * s_iSB);
                }
                __syncthreads();
                nc.s = s_s;
                k1 = 1.0 - (double)nc.s;
                for (int i = tid; i < kTreeWarps * kTreeGroups; i += kTreeThreads)
                    s_mass[i] = fmaxf(0.f, (float)((double)s_mass[i] + k1 * (double)s_mass2[i]));
                if (lane == 0) s_red[warp][0] = fmax(0.0, s_red[warp][2] + k1 * s_red[warp][3]);
                __syncthreads();
            }
            if (warp == 0) {
                // the masses of the cluster's CTAs, their total, the threshold
                const double Mr = lane >= cs ? 0.0
                                  : first_rec ? fmax(0.0, ld_cluster_f64(&s_slot[par][2], lane) +
                                                              k1 * ld_cluster_f64(&s_slot[par][3], lane))
                                              : ld_cluster_f64(&s_slot[par][0], lane);
                const double Z = warp_sum_d(Mr);
                const double thr = s_us[cur] * Z;
                // the CTA whose slice holds the crossing, then (in it) the warp
                double base = 0.0;
                const int R = crossing_lane(Mr, 0.0, thr, lane, base);
                int W = -1;
                if (R == rank) {
                    double wb = base;
                    W = crossing_lane(lane < kTreeWarps ? s_red[lane][0] : 0.0, base, thr, lane, wb);
                    base = wb;
                }
                if (lane == 0) {
                    s_again = 0;
                    if (!(Z > 0.0) && mode != kTreeModeP) {  // no residual mass: p
                        s_s = 0.f;
                        s_again = 1;
                    }
                    s_R = R < 0 ? 0 : R;
                    s_W = W;
                    s_base = base;
                    s_thr = thr;
                    s_emit = V - 1;  // no mass at all
                }
            }
            par ^= 1;
            __syncthreads();
            first_rec = false;
            if (!s_again) break;
            nc.s = s_s;
        }
        const int mode = nc.s > 0.f ? kTreeModeThr : kTreeModeP;
        if (rank == s_R && s_W >= 0 && warp == 0) {
            const bool use_stage = staged && !s_nostage;
            if (use_stage)  // warp W's copy completed before its pass: acquire it here
                mbar_wait_bounded(&s_tbar[s_W], (stagings - 1u) & 1u, kWaitLimitNs);
            const int tok = tree_find<DT, VEC>(rowt, rowd, use_stage ? stt : nullptr,
                                               use_stage ? std_ : nullptr, V, rank, cs, nc, mode,
                                               s_mass, s_W, s_base, s_thr, lane);
            if (lane == 0 && tok >= 0) s_emit = tok;
        }
        __syncthreads();
        if (tid == 0 && rank == s_R) out[depth] = s_emit;
        if (tid == 0 && rank == 0) {
            for (int i = depth + 1; i < N; ++i) out[i] = -1;
            for (int i = depth; i < N; ++i) nodes[i] = -1;
            P.accept_len[b] = depth;
        }
        cluster_sync_all();  // no CTA leaves while another may read its slots
        return;
    }
}

// ------------------------------------------------------------------ load-aware schedule

constexpr int kBudgetThreads = 1024;
constexpr long long kBudgetMaxN = 1 << 22;  // positions B * K one CTA selects from

// Survival key of position (b, k): the float bits of the running product of
// clamped max-probabilities (non-negative, so ordered as integers) above the
// complemented flat index, so that larger keys survive more and ties go to the
// lower (b, k).  All keys differ.
__device__ __forceinline__ unsigned long long survival_key(float s, long long i) {
    return ((unsigned long long)__float_as_uint(s) << 32) | (0xFFFFFFFFull - (unsigned long long)i);
}
__device__ __forceinline__ float clamp_prob(float c) {
    if (!(c >= 0.0f)) c = 0.0f;  // NaN too
    return c > 1.0f ? 1.0f : c;
}

// One CTA: the budget-th largest survival key by an 8-pass byte radix select
// (keys recomputed each pass), then each request's verify length = the number
// of its positions at or above that key (a prefix, since survival never grows
// along a request).
__global__ void __launch_bounds__(kBudgetThreads) sv_schedule_budget(const float *__restrict__ mp,
                                                                    int B, int K, long long budget,
                                                                    int32_t *__restrict__ out) {
    __shared__ unsigned hist[256];
    __shared__ unsigned long long s_prefix;
    __shared__ long long s_rem;
    const int tid = threadIdx.x;
    const long long n = (long long)B * K;
    if (budget <= 0 || budget >= n) {
        for (int b = tid; b < B; b += kBudgetThreads) out[b] = budget <= 0 ? 0 : K;
        return;
    }
    if (tid == 0) {
        s_prefix = 0ull;
        s_rem = budget;  // rank still to place (1-based) among the matching keys
    }
    unsigned long long mask = 0ull;
    for (int pass = 7; pass >= 0; --pass) {
        for (int i = tid; i < 256; i += kBudgetThreads) hist[i] = 0u;
        __syncthreads();
        const unsigned long long prefix = s_prefix;
        const int sh = pass * 8;
        for (int b = tid; b < B; b += kBudgetThreads) {
            float s = 1.0f;
            for (int k = 0; k < K; ++k) {
                s = __fmul_rn(s, clamp_prob(mp[(size_t)b * K + k]));
                const unsigned long long key = survival_key(s, (long long)b * K + k);
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & 0xFFu], 1u);
            }
        }
        __syncthreads();
        if (tid == 0) {
            long long rem = s_rem;
            int d = 255;
            for (; d > 0; --d) {
                if ((long long)hist[d] >= rem) break;
                rem -= hist[d];
            }
            s_rem = rem;
            s_prefix = prefix | ((unsigned long long)d << sh);
        }
        mask |= 0xFFull << sh;
        __syncthreads();
    }
    const unsigned long long tau = s_prefix;  // the budget-th largest key
    for (int b = tid; b < B; b += kBudgetThreads) {
        float s = 1.0f;
        int L = 0;
        for (int k = 0; k < K; ++k) {
            s = __fmul_rn(s, clamp_prob(mp[(size_t)b * K + k]));
            if (survival_key(s, (long long)b * K + k) >= tau) L = k + 1;
            else break;
        }
        out[b] = L;
    }
}

// ------------------------------------------------------------------ LM head (epilogues)

// Statistics epilogue of the LM-head GEMM: the same per-row statistics the
// streaming pass produces, taken from the fp32 accumulators of a 128 x 256
// tile instead of a logit row in memory ("speculative decoding от черновика до
// проверки" (braintools.ru), "Как это работает", step 2: the target scores
// all drafts in one pass, whose last step is this product).  Row r of the
// product is slot slot0 + r % rows_per_req of request r / rows_per_req; per
// (row, tile) one partial {max, sum 2^((z - max) log2(e)/T), -1} (sampled
// request) or {max, 0, lowest index of the max} (greedy request), and the
// logit at the row's draft token when the tile holds it.
struct LmStatsEpi {
    float4 *part;
    float *gz;
    const int32_t *tokens;
    const float *temperature;
    int npart, nslot, K;
    int rows_per_req[2], slot0[2], tok_off[2];  // per row segment (target rows, draft rows)
    __device__ __forceinline__ void row(int seg, int r, bool valid, int n0, int V,
                                        uint32_t taddr) const {
        int b = 0, slot = 0, x = -1;
        bool greedy = true;
        float c = 0.f;
        if (valid) {  // (selects, not indexing: the functor stays in registers)
            const int rpr = seg ? rows_per_req[1] : rows_per_req[0];
            b = r / rpr;
            slot = (seg ? slot0[1] : slot0[0]) + (r - b * rpr);
            const int tk = slot - (seg ? tok_off[1] : tok_off[0]);  // the draft token this row scores
            if (tk >= 0 && tk < K) x = tokens[(size_t)b * K + tk];
            const float T = temperature[b];
            greedy = !(isfinite(T) && T >= FLT_MIN);
            if (!greedy) c = __fdiv_rn(kLog2EHi, T);  // the statistics pass's factor
        }
        float m = -INFINITY, s = 0.f, g = 0.f;
        int am = INT_MAX;
        bool have_g = false;
        const unsigned long long c2 = f2u(make_float2(c, c));
#pragma unroll 1
        for (int j = 0; j < kLmBN / 32; ++j) {
            float v[32];
            __syncwarp();
            tmem_ld32(taddr + (uint32_t)(j * 32), v);
            const int nb = n0 + j * 32;
            if (nb + 32 > V) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (nb + i >= V) v[i] = -INFINITY;
            }
            if (x >= nb && x < nb + 32) {  // a binary select tree, no indexed local copy of v
                const int o = x - nb;
                float t16[16], t8[8], t4[4], t2[2];
#pragma unroll
                for (int i = 0; i < 16; ++i) t16[i] = (o & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
                for (int i = 0; i < 8; ++i) t8[i] = (o & 2) ? t16[2 * i + 1] : t16[2 * i];
#pragma unroll
                for (int i = 0; i < 4; ++i) t4[i] = (o & 4) ? t8[2 * i + 1] : t8[2 * i];
#pragma unroll
                for (int i = 0; i < 2; ++i) t2[i] = (o & 8) ? t4[2 * i + 1] : t4[2 * i];
                g = (o & 16) ? t2[1] : t2[0];
                have_g = true;
            }
            float cm = v[0];
#pragma unroll
            for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
            if (greedy) {
                if (cm > m) {  // chunks come in increasing index order
                    int idx = 31;
#pragma unroll
                    for (int i = 31; i >= 0; --i)
                        if (v[i] == cm) idx = i;
                    m = cm;
                    am = nb + idx;
                }
            } else if (cm > -INFINITY) {
                if (cm > m) {
                    if (m > -INFINITY) s *= ex2((m - cm) * c);
                    m = cm;
                }
                const unsigned long long m2 = f2u(make_float2(m, m));
                unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    f32x2_exp_acc(__float_as_uint(v[i]), __float_as_uint(v[i + 1]), m2, c2, a0);
                    f32x2_exp_acc(__float_as_uint(v[i + 2]), __float_as_uint(v[i + 3]), m2, c2, a1);
                }
                const float2 t = add2(u2f(a0), u2f(a1));
                s += t.x + t.y;
            }
        }
        if (valid) {
            part[((size_t)b * nslot + slot) * npart + n0 / kLmBN] =
                greedy ? make_float4(m, 0.f, __int_as_float(am), 0.f)
                       : make_float4(m, s, __int_as_float(-1), 0.f);
            if (have_g) gz[(size_t)b * nslot + slot] = g;
        }
    }
};

// Store epilogue: the rows themselves (fp32), for the few rows the sampler
// draws from, recomputed after the decisions.
struct LmStoreEpi {
    float *out[2];  // [rows, V] per row segment
    __device__ __forceinline__ void row(int seg, int r, bool valid, int n0, int V,
                                        uint32_t taddr) const {
        float *o = (seg ? out[1] : out[0]) + (size_t)r * (size_t)V;
#pragma unroll 1
        for (int j = 0; j < kLmBN / 32; ++j) {
            float v[32];
            __syncwarp();
            tmem_ld32(taddr + (uint32_t)(j * 32), v);
            const int nb = n0 + j * 32;
            if (!valid) continue;
            if (nb + 32 <= V && (V & 3) == 0) {
                float4 *o4 = reinterpret_cast<float4 *>(o + nb);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    o4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            } else {
                for (int i = 0; i < 32; ++i)
                    if (nb + i < V) o[nb + i] = v[i];
            }
        }
    }
};

// The hidden states of each sampled request's draw rows, packed by its entry
// li in the sampled-request list (target row a or L; draft row a for a
// residual draw, zeros for a bonus draw), for the recompute of those rows:
// target row at hct + li * stride rows, draft row at hcd + li * stride rows.
__global__ void __launch_bounds__(256) lm_gather(Params P, const uint16_t *ht, const uint16_t *hd,
                                                  int d, uint16_t *hct, uint16_t *hcd, int stride) {
    pdl_wait();  // the list comes from sv_decide
    pdl_trigger();
    const int li = blockIdx.x;
    if (li >= *P.samp_count) return;
    const SampInfo si = P.samp_list[li];
    const int K = P.K, nv = d / 8;
    const uint4 *st = reinterpret_cast<const uint4 *>(ht + ((size_t)si.b * (K + 1) + si.slot_t) * d);
    uint4 *dt = reinterpret_cast<uint4 *>(hct + (size_t)li * stride * d);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) dt[i] = st[i];
    uint4 *dd = reinterpret_cast<uint4 *>(hcd + (size_t)li * stride * d);
    if (si.mode == 1) {
        const uint4 *sd =
            reinterpret_cast<const uint4 *>(hd + ((size_t)si.b * K + (si.slot_d - K - 1)) * d);
        for (int i = threadIdx.x; i < nv; i += blockDim.x) dd[i] = sd[i];
    } else {
        for (int i = threadIdx.x; i < nv; i += blockDim.x) dd[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// ------------------------------------------------------------------ host side

struct Layout {
    size_t req, row_count, rows, part, sub, sexact, samp_list, samp_count, ee_done, mp, vlen, total;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int chunk_elems_for(spec_dtype_t dt) {
    return dt == SPEC_DTYPE_BF16 ? chunk_elems<kBF16>() : chunk_elems<kF32>();
}

static bool sizes_ok(int B, int K, int V) {
    return B >= 1 && B < (1 << 24) && K >= 1 && K <= SPEC_MAX_K && V >= 2 && V <= SPEC_MAX_V;
}

static size_t nchunk_for(int V, spec_dtype_t dt) {
    return (size_t)((V + chunk_elems_for(dt) - 1) / chunk_elems_for(dt));
}

static size_t npart_for(int V, spec_dtype_t dt) {
    const int pe = dt == SPEC_DTYPE_BF16 ? p1_item_elems<kBF16>() : p1_item_elems<kF32>();
    return (size_t)((V + pe - 1) / pe);
}

// Work items are indexed with 32-bit integers.
static bool items_fit(int B, int K, int V, spec_dtype_t dt) {
    return (size_t)B * (size_t)(2 * K + 1) * nchunk_for(V, dt) < ((size_t)1 << 31);
}

static Layout layout(int B, int K, int V, spec_dtype_t dt) {
    Layout L{};
    const size_t nchunk = nchunk_for(V, dt);
    const size_t nslot = (size_t)(2 * K + 1);
    size_t off = 0;
    L.req = off; off = align256(off + sizeof(ReqInfo) * (size_t)B);
    L.row_count = off; off = align256(off + sizeof(int));
    L.rows = off; off = align256(off + sizeof(int4) * (size_t)B * nslot);
    L.part = off; off = align256(off + sizeof(float4) * (size_t)B * nslot * npart_for(V, dt));
    L.sub = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.sexact = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.samp_list = off; off = align256(off + sizeof(SampInfo) * (size_t)B);
    L.samp_count = off; off = align256(off + sizeof(int));
    L.ee_done = off; off = align256(off + sizeof(int) * (size_t)B);
    L.mp = off; off = align256(off + sizeof(float) * (size_t)B * (size_t)K);
    L.vlen = off; off = align256(off + sizeof(int) * (size_t)B);
    L.total = off;
    return L;
}

struct DevInfo {
    int sms = 0;
    int occ_p1[2][2] = {{0, 0}, {0, 0}};
    int occ_sample[2][2] = {{0, 0}, {0, 0}};
    int occ_decide[2] = {0, 0};  // resident sv_decide CTAs per SM at the default register budget
    bool walk_smem[2][2] = {{false, false}, {false, false}};  // tree walk's shared-memory limit raised
    bool lm_ready = false;  // LM-head GEMM's shared-memory limit raised
    bool ok = false;
};

static DevInfo g_dev[64];
constexpr size_t kP1Smem = sizeof(P1Shared);
constexpr size_t kSSmem = sizeof(SShared);

template <int DT, bool VEC>
static bool setup_kernels(DevInfo &d) {
    const size_t smem1 = VEC ? kP1Smem : 0, smem2 = VEC ? kSSmem : 0;
    if (VEC && (cudaFuncSetAttribute(sv_pass1<DT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem1) != cudaSuccess ||
                cudaFuncSetAttribute(sv_sample<DT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem2) != cudaSuccess ||
                cudaFuncSetAttribute(sv_pass1<DT, VEC, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess ||
                cudaFuncSetAttribute(sv_sample<DT, VEC, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess))
        return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_pass1<DT, VEC>, kP1Warps * 32, smem1) !=
        cudaSuccess)
        return false;
    d.occ_p1[DT][VEC] = o > 0 ? o : 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_sample<DT, VEC>, kSWarps * 32, smem2) !=
        cudaSuccess)
        return false;
    d.occ_sample[DT][VEC] = o > 0 ? o : 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_decide<DT>, kThreads, 0) != cudaSuccess)
        return false;
    d.occ_decide[DT] = o > 0 ? o : 1;
    return true;
}

// The decision kernel for a batch: one CTA per request, all resident at once
// when the default register budget allows it, else the build cut to 4 CTAs
// per SM.
template <int DT>
static void (*decide_kernel(const DevInfo &d, int B))(Params) {
    return (long long)B > (long long)d.occ_decide[DT] * d.sms ? sv_decide<DT, 4> : sv_decide<DT>;
}

static DevInfo *dev_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    DevInfo &d = g_dev[dev];
    if (!d.ok) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        if (!setup_kernels<kF32, false>(d) || !setup_kernels<kF32, true>(d) ||
            !setup_kernels<kBF16, false>(d) || !setup_kernels<kBF16, true>(d))
            return nullptr;
        d.sms = sms;
        d.ok = true;
    }
    return &d;
}

static cudaEvent_t g_prof_start = nullptr, g_prof_end = nullptr;
constexpr int kKernelsPerVerify = 5;

// Launch that may begin while the previous kernel of the stream is still
// running (programmatic dependent launch): the kernel does its independent
// set-up, then griddepcontrol.wait blocks until the previous kernel has
// completed and its writes are visible.
static void launch_dependent(void (*kernel)(Params), int grid, int block, size_t smem,
                             cudaStream_t s, const Params &P) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, P);
}

template <int DT, bool VEC>
static void launch_all(const Params &P, const DevInfo &d, cudaStream_t s) {
    // sv_prep is an ordinary launch: it starts only after all earlier work of
    // the stream, so the workspace of a previous call is free again.
    sv_prep<<<1, prep_threads(P.B), 0, s>>>(P);
    if (g_prof_start) cudaEventRecord(g_prof_start, s);
    launch_dependent(g_diag_timeout ? sv_pass1<DT, VEC, true> : sv_pass1<DT, VEC>,
                     d.sms * d.occ_p1[DT][VEC], kP1Warps * 32, VEC ? kP1Smem : 0, s, P);
    if (g_prof_end) cudaEventRecord(g_prof_end, s);
    launch_dependent(decide_kernel<DT>(d, P.B), P.B, kThreads, 0, s, P);
    // the sampled requests are known only on the device: enough warps for all
    // of them, at most one full wave
    long long g2 = (long long)d.sms * d.occ_sample[DT][VEC];
    const long long g2_need = ((long long)P.B * P.nchunk + kSWarps - 1) / kSWarps;
    if (g2 > g2_need) g2 = g2_need;
    launch_dependent(g_diag_timeout ? sv_sample<DT, VEC, true> : sv_sample<DT, VEC>, (int)g2,
                     kSWarps * 32, VEC ? kSSmem : 0, s, P);
    launch_dependent(sv_find<DT, VEC>, P.B, kFindWarps * 32, 0, s,
                     P);
}

// Early exit: the positions in two waves, [0, W) then [W, K).  A wave lists
// the rows its still-open requests need, streams them and decides; a request
// whose first rejection (or whose L) falls in the first wave needs no row of
// the second.  Each wave's sv_prep is an ordinary launch, so it starts after
// the previous wave's decisions.  The sampler and inverse CDF run once.
template <int DT, bool VEC>
static void launch_waves(const Params &P0, const DevInfo &d, cudaStream_t s, int W) {
    Params P = P0;
    const int nw = (W > 0 && W < P.K) ? 2 : 1;
    for (int w = 0; w < nw; ++w) {
        P.k0 = w == 0 ? 0 : W;
        P.k1 = (w == 0 && nw == 2) ? W : P.K;
        sv_prep<<<1, prep_threads(P.B), 0, s>>>(P);
        launch_dependent(sv_pass1<DT, VEC>, d.sms * d.occ_p1[DT][VEC], kP1Warps * 32,
                         VEC ? kP1Smem : 0, s, P);
        launch_dependent(decide_kernel<DT>(d, P.B), P.B, kThreads, 0, s, P);
    }
    long long g2 = (long long)d.sms * d.occ_sample[DT][VEC];
    const long long g2_need = ((long long)P.B * P.nchunk + kSWarps - 1) / kSWarps;
    if (g2 > g2_need) g2 = g2_need;
    launch_dependent(sv_sample<DT, VEC>, (int)g2, kSWarps * 32, VEC ? kSSmem : 0, s, P);
    launch_dependent(sv_find<DT, VEC>, P.B, kFindWarps * 32, 0, s,
                     P);
}

// Host-side checks of the step's arguments and the Params they give (the
// workspace cut into its regions).  Nothing is launched.
static spec_status_t step_params(Params &P, const void *target_logits, const void *draft_logits,
                                 spec_dtype_t dtype, const int32_t *draft_tokens,
                                 const int32_t *verify_len, const float *temperature,
                                 uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                 int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                 uint32_t *dev_status, Layout &L) {
    if (!sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    if (!items_fit(B, K, V, dtype)) return SPEC_ERR_UNSUPPORTED;
    if (!target_logits || !draft_logits || !draft_tokens || !temperature || !out_tokens ||
        !accept_len)
        return SPEC_ERR_INVALID_ARG;
    if (((uintptr_t)target_logits & 15u) || ((uintptr_t)draft_logits & 15u))
        return SPEC_ERR_INVALID_ARG;
    L = layout(B, K, V, dtype);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    P = Params{};
    P.tgt = static_cast<const char *>(target_logits);
    P.drf = static_cast<const char *>(draft_logits);
    P.tokens = draft_tokens;
    P.verify_len = verify_len;
    P.temperature = temperature;
    P.seed = seed;
    P.B = B;
    P.K = K;
    P.V = V;
    P.nchunk = (int)nchunk_for(V, dtype);
    P.npart = (int)npart_for(V, dtype);
    P.nslot = 2 * K + 1;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    char *ws = static_cast<char *>(workspace);
    P.req = reinterpret_cast<ReqInfo *>(ws + L.req);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    P.sub = reinterpret_cast<float4 *>(ws + L.sub);
    P.sexact = reinterpret_cast<float4 *>(ws + L.sexact);
    P.samp_list = reinterpret_cast<SampInfo *>(ws + L.samp_list);
    P.samp_count = reinterpret_cast<int *>(ws + L.samp_count);
    P.k0 = 0;
    P.k1 = K;
    P.ee_done = nullptr;
    return SPEC_OK;
}

static bool vec_rows(int V, spec_dtype_t dtype) {
    return ((size_t)V * (size_t)(dtype == SPEC_DTYPE_BF16 ? 2 : 4)) % 16u == 0;
}

// The five kernels of one step, for the logits' dtype and row alignment.
static void launch_step(const Params &P, const DevInfo &d, cudaStream_t s, spec_dtype_t dtype,
                        bool vec) {
    if (dtype == SPEC_DTYPE_BF16) {
        if (vec) launch_all<kBF16, true>(P, d, s);
        else launch_all<kBF16, false>(P, d, s);
    } else {
        if (vec) launch_all<kF32, true>(P, d, s);
        else launch_all<kF32, false>(P, d, s);
    }
}

static spec_status_t verify_impl(const void *target_logits, const void *draft_logits,
                                 spec_dtype_t dtype, const int32_t *draft_tokens,
                                 const int32_t *verify_len, const float *temperature,
                                 uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                 int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                 uint32_t *dev_status, double *row_stats, double *probs,
                                 void *stream, int first_wave = 0) {
    if (first_wave < 0) return SPEC_ERR_INVALID_ARG;
    Params P;
    Layout L;
    const spec_status_t st = step_params(P, target_logits, draft_logits, dtype, draft_tokens,
                                         verify_len, temperature, seed, B, K, V, out_tokens,
                                         accept_len, workspace, workspace_bytes, dev_status, L);
    if (st != SPEC_OK) return st;
    DevInfo *d = dev_info();
    if (!d) return SPEC_ERR_CUDA;
    const bool vec = vec_rows(V, dtype);
    P.dbg_rows = row_stats;
    P.dbg_probs = probs;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (first_wave > 0) {
        P.ee_done = reinterpret_cast<int *>(static_cast<char *>(workspace) + L.ee_done);
        P.dbg_rows = nullptr;
        P.dbg_probs = nullptr;
        if (dtype == SPEC_DTYPE_BF16) {
            if (vec) launch_waves<kBF16, true>(P, *d, s, first_wave);
            else launch_waves<kBF16, false>(P, *d, s, first_wave);
        } else {
            if (vec) launch_waves<kF32, true>(P, *d, s, first_wave);
            else launch_waves<kF32, false>(P, *d, s, first_wave);
        }
    } else {
        launch_step(P, *d, s, dtype, vec);
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Confidence pass of the draft rows: every draft row of every sampled request
// through the statistics pass (its partials stay in the workspace, in the
// slots the step's decision kernel reads), then max_v q per row.
static void launch_confidence(const Params &P, const DevInfo &d, cudaStream_t s,
                              spec_dtype_t dtype, bool vec, float *maxprob) {
    sv_conf_rows<<<1, kPrepThreads, 0, s>>>(P);
    const int g1 = d.sms * d.occ_p1[dtype == SPEC_DTYPE_BF16 ? kBF16 : kF32][vec ? 1 : 0];
    if (dtype == SPEC_DTYPE_BF16) {
        if (vec) launch_dependent(sv_pass1<kBF16, true>, g1, kP1Warps * 32, kP1Smem, s, P);
        else launch_dependent(sv_pass1<kBF16, false>, g1, kP1Warps * 32, 0, s, P);
    } else {
        if (vec) launch_dependent(sv_pass1<kF32, true>, g1, kP1Warps * 32, kP1Smem, s, P);
        else launch_dependent(sv_pass1<kF32, false>, g1, kP1Warps * 32, 0, s, P);
    }
    const long long rows = (long long)P.B * P.K;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, sv_conf_out, P, maxprob);
}

// ------------------------------------------------------------------ LM head (host)

static size_t npart_lm(int V) { return (size_t)((V + kLmBN - 1) / kLmBN); }

struct LmLayout {
    size_t req, row_count, rows, part, sub, sexact, samp_list, samp_count, gz, hc, crow, total;
};

static LmLayout layout_lm(int B, int K, int V, int d) {
    LmLayout L{};
    const size_t nslot = (size_t)(2 * K + 1), nchunk = nchunk_for(V, SPEC_DTYPE_F32);
    size_t off = 0;
    L.req = off; off = align256(off + sizeof(ReqInfo) * (size_t)B);
    L.row_count = off; off = align256(off + sizeof(int));
    L.rows = off; off = align256(off + sizeof(int4) * (size_t)B * nslot);
    L.part = off; off = align256(off + sizeof(float4) * (size_t)B * nslot * npart_lm(V));
    L.sub = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.sexact = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.samp_list = off; off = align256(off + sizeof(SampInfo) * (size_t)B);
    L.samp_count = off; off = align256(off + sizeof(int));
    L.gz = off; off = align256(off + sizeof(float) * (size_t)B * nslot);
    L.hc = off; off = align256(off + 2 * 2 * (size_t)B * (size_t)d);    // 2B hidden rows, bf16
    L.crow = off; off = align256(off + 4 * 2 * (size_t)B * (size_t)V);  // 2B logit rows, fp32
    L.total = off;
    return L;
}

static bool lm_sizes_ok(int B, int K, int V, int d) {
    return sizes_ok(B, K, V) && d >= kLmBK && d % kLmBK == 0 && d <= (1 << 16) &&
           (size_t)B * (size_t)(K + 1) < ((size_t)1 << 31) && (V % 4) == 0 &&
           (size_t)B * (size_t)(2 * K + 1) * nchunk_for(V, SPEC_DTYPE_F32) < ((size_t)1 << 31);
}

// A 2D tensor map over a row-major bf16 matrix [rows, cols] with boxes of
// 64 columns (128 bytes, the swizzle span) by box_rows rows, 128-byte swizzle,
// out-of-range elements read as zero.
static bool make_tmap_bf16(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kLmBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One product over up to two row segments (rows [0, M0) of tA0, rows [0, M1)
// of tA1) against the weights of tB; M0 is capped on the device at
// mult * *M_dev when M_dev is given.
template <class Epi>
static cudaError_t launch_lm_gemm(const CUtensorMap &tA0, const CUtensorMap &tA1,
                                  const CUtensorMap &tB, int M0, int M1, const int *M_dev,
                                  int mult, int V, int d, const Epi &epi, uint32_t *status,
                                  const DevInfo &dv, cudaStream_t s) {
    const long long tiles = ((long long)(M0 + kLmBM - 1) / kLmBM + (M1 + kLmBM - 1) / kLmBM) *
                            ((V + kLmBN - 1) / kLmBN);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < dv.sms ? (tiles > 0 ? tiles : 1) : dv.sms));
    cfg.blockDim = dim3(kLmThreads);
    cfg.dynamicSmemBytes = kLmSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lm_gemm<Epi>, tA0, tA1, tB, M0, M1, M_dev, mult, V, d, epi,
                              status, g_diag_timeout ? 1 : 0, kDiagWaitNs);
}

static bool lm_setup(DevInfo &d) {
    if (d.lm_ready) return true;
    if (cudaFuncSetAttribute(lm_gemm<LmStatsEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLmSmem) != cudaSuccess ||
        cudaFuncSetAttribute(lm_gemm<LmStoreEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLmSmem) != cudaSuccess)
        return false;
    d.lm_ready = true;
    return true;
}

} // namespace sv

namespace sv {
// Host-to-device copies of byte ranges, each merged into the previous one when
// it continues it in both memories; `total` counts the bytes enqueued.
struct H2DRuns {
    cudaStream_t s = nullptr;
    const char *src = nullptr;
    char *dst = nullptr;
    size_t n = 0, total = 0;
    bool ok = true;
    void add(const void *from, void *to, size_t bytes) {
        const char *f = static_cast<const char *>(from);
        char *t = static_cast<char *>(to);
        if (!bytes) return;
        if (n && f == src + n && t == dst + n) {
            n += bytes;
            return;
        }
        flush();
        src = f;
        dst = t;
        n = bytes;
    }
    void flush() {
        if (!n) return;
        if (cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s) != cudaSuccess) ok = false;
        total += n;
        n = 0;
    }
};
}  // namespace sv

extern "C" {

size_t spec_verify_workspace_bytes(int B, int K, int V, spec_dtype_t dtype) {
    if (!sv::sizes_ok(B, K, V)) return 0;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
    return sv::layout(B, K, V, dtype).total;
}

spec_status_t spec_verify(const void *target_logits, const void *draft_logits,
                          spec_dtype_t dtype, const int32_t *draft_tokens,
                          const int32_t *verify_len, const float *temperature, uint64_t seed,
                          int B, int K, int V, int32_t *out_tokens, int32_t *accept_len,
                          void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                          void *stream) {
    return sv::verify_impl(target_logits, draft_logits, dtype, draft_tokens, verify_len,
                           temperature, seed, B, K, V, out_tokens, accept_len, workspace,
                           workspace_bytes, dev_status, nullptr, nullptr, stream);
}

spec_status_t spec_verify_debug(const void *target_logits, const void *draft_logits,
                                spec_dtype_t dtype, const int32_t *draft_tokens,
                                const int32_t *verify_len, const float *temperature,
                                uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                uint32_t *dev_status, double *row_stats, double *probs,
                                void *stream) {
    return sv::verify_impl(target_logits, draft_logits, dtype, draft_tokens, verify_len,
                           temperature, seed, B, K, V, out_tokens, accept_len, workspace,
                           workspace_bytes, dev_status, row_stats, probs, stream);
}

spec_status_t spec_verify_early_exit(const void *target_logits, const void *draft_logits,
                                     spec_dtype_t dtype, const int32_t *draft_tokens,
                                     const int32_t *verify_len, const float *temperature,
                                     uint64_t seed, int B, int K, int V, int first_wave,
                                     int32_t *out_tokens, int32_t *accept_len, void *workspace,
                                     size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    if (first_wave < 1) return SPEC_ERR_INVALID_ARG;
    return sv::verify_impl(target_logits, draft_logits, dtype, draft_tokens, verify_len,
                           temperature, seed, B, K, V, out_tokens, accept_len, workspace,
                           workspace_bytes, dev_status, nullptr, nullptr, stream, first_wave);
}

spec_status_t spec_draft_confidence(const void *draft_logits, spec_dtype_t dtype,
                                    const float *temperature, int B, int K, int V,
                                    float *maxprob, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (!sv::sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    if (!sv::items_fit(B, K, V, dtype)) return SPEC_ERR_UNSUPPORTED;
    if (!draft_logits || !temperature || !maxprob) return SPEC_ERR_INVALID_ARG;
    if ((uintptr_t)draft_logits & 15u) return SPEC_ERR_INVALID_ARG;
    const sv::Layout L = sv::layout(B, K, V, dtype);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    sv::DevInfo *d = sv::dev_info();
    if (!d) return SPEC_ERR_CUDA;
    sv::Params P{};
    P.tgt = static_cast<const char *>(draft_logits);  // only draft rows are listed
    P.drf = static_cast<const char *>(draft_logits);
    P.temperature = temperature;
    P.B = B;
    P.K = K;
    P.V = V;
    P.nchunk = (int)sv::nchunk_for(V, dtype);
    P.npart = (int)sv::npart_for(V, dtype);
    P.nslot = 2 * K + 1;
    P.k0 = 0;
    P.k1 = K;
    char *ws = static_cast<char *>(workspace);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    sv::launch_confidence(P, *d, static_cast<cudaStream_t>(stream), dtype, sv::vec_rows(V, dtype),
                          maxprob);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_scheduled(const void *target_logits, const void *draft_logits,
                                    spec_dtype_t dtype, const int32_t *draft_tokens,
                                    const float *temperature, uint64_t seed, int B, int K, int V,
                                    const float *draft_maxprob, spec_sched_mode_t mode,
                                    float threshold, long long budget, float *maxprob_out,
                                    int32_t *verify_len_out, int32_t *out_tokens,
                                    int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                    uint32_t *dev_status, void *stream) {
    if (mode != SPEC_SCHED_THRESHOLD && mode != SPEC_SCHED_BUDGET) return SPEC_ERR_INVALID_ARG;
    sv::Params P;
    sv::Layout L;
    const spec_status_t st = sv::step_params(P, target_logits, draft_logits, dtype, draft_tokens,
                                             nullptr, temperature, seed, B, K, V, out_tokens,
                                             accept_len, workspace, workspace_bytes, dev_status, L);
    if (st != SPEC_OK) return st;
    if (mode == SPEC_SCHED_BUDGET && (long long)B * K > sv::kBudgetMaxN) return SPEC_ERR_UNSUPPORTED;
    sv::DevInfo *d = sv::dev_info();
    if (!d) return SPEC_ERR_CUDA;
    const bool vec = sv::vec_rows(V, dtype);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const float *mp = draft_maxprob;
    if (!mp) {  // confidences from the draft rows; their statistics serve the step too
        float *out = maxprob_out ? maxprob_out : reinterpret_cast<float *>(ws + L.mp);
        sv::launch_confidence(P, *d, s, dtype, vec, out);
        mp = out;
        P.draft_ready = 1;
    }
    if (mode == SPEC_SCHED_THRESHOLD) {  // sv_prep takes each length from the product itself
        P.sched_mp = mp;
        P.sched_thr = threshold;
        P.vlen_out = verify_len_out;
    } else {
        int32_t *vl = verify_len_out ? verify_len_out : reinterpret_cast<int32_t *>(ws + L.vlen);
        sv::sv_schedule_budget<<<1, sv::kBudgetThreads, 0, s>>>(mp, B, K, budget, vl);
        P.verify_len = vl;
    }
    sv::launch_step(P, *d, s, dtype, vec);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

size_t spec_lmhead_workspace_bytes(int B, int K, int V, int d) {
    if (!sv::lm_sizes_ok(B, K, V, d)) return 0;
    return sv::layout_lm(B, K, V, d).total;
}

spec_status_t spec_verify_lmhead(const void *hidden_target, const void *hidden_draft,
                                 const void *w_target, const void *w_draft, int d,
                                 const int32_t *draft_tokens, const int32_t *verify_len,
                                 const float *temperature, uint64_t seed, int B, int K, int V,
                                 int32_t *out_tokens, int32_t *accept_len, void *workspace,
                                 size_t workspace_bytes, uint32_t *dev_status, double *row_stats,
                                 double *probs, void *stream) {
    if (!sv::lm_sizes_ok(B, K, V, d)) return SPEC_ERR_INVALID_ARG;
    if (!hidden_target || !hidden_draft || !w_target || !w_draft || !draft_tokens ||
        !temperature || !out_tokens || !accept_len)
        return SPEC_ERR_INVALID_ARG;
    if (((uintptr_t)hidden_target & 15u) || ((uintptr_t)hidden_draft & 15u) ||
        ((uintptr_t)w_target & 15u) || ((uintptr_t)w_draft & 15u))
        return SPEC_ERR_INVALID_ARG;
    const sv::LmLayout L = sv::layout_lm(B, K, V, d);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    sv::DevInfo *dv = sv::dev_info();
    if (!dv || !sv::lm_setup(*dv)) return SPEC_ERR_CUDA;
    char *ws = static_cast<char *>(workspace);
    // the drafter shares the target's head: one product over both row sets
    // (the weights stream once), and one recompute over interleaved rows
    const bool shared = w_target == w_draft;
    uint16_t *hc = reinterpret_cast<uint16_t *>(ws + L.hc);
    float *crow = reinterpret_cast<float *>(ws + L.crow);
    CUtensorMap tHt, tHd, tWt, tWd, tC0, tC1;
    if (!sv::make_tmap_bf16(&tHt, hidden_target, (uint64_t)B * (K + 1), (uint64_t)d, sv::kLmBM) ||
        !sv::make_tmap_bf16(&tHd, hidden_draft, (uint64_t)B * K, (uint64_t)d, sv::kLmBM) ||
        !sv::make_tmap_bf16(&tWt, w_target, (uint64_t)V, (uint64_t)d, sv::kLmBN) ||
        !sv::make_tmap_bf16(&tWd, w_draft, (uint64_t)V, (uint64_t)d, sv::kLmBN) ||
        !sv::make_tmap_bf16(&tC0, hc, (uint64_t)(shared ? 2 * B : B), (uint64_t)d, sv::kLmBM) ||
        !sv::make_tmap_bf16(&tC1, hc + (size_t)B * d, (uint64_t)B, (uint64_t)d, sv::kLmBM))
        return SPEC_ERR_CUDA;
    sv::Params P{};
    P.tgt = ws + L.crow;  // no logit row is read in place on this path
    P.drf = ws + L.crow;
    P.tokens = draft_tokens;
    P.verify_len = verify_len;
    P.temperature = temperature;
    P.seed = seed;
    P.B = B;
    P.K = K;
    P.V = V;
    P.nchunk = (int)sv::nchunk_for(V, SPEC_DTYPE_F32);
    P.npart = (int)sv::npart_lm(V);
    P.nslot = 2 * K + 1;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    P.dbg_rows = row_stats;
    P.dbg_probs = probs;
    P.req = reinterpret_cast<sv::ReqInfo *>(ws + L.req);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    P.sub = reinterpret_cast<float4 *>(ws + L.sub);
    P.sexact = reinterpret_cast<float4 *>(ws + L.sexact);
    P.samp_list = reinterpret_cast<sv::SampInfo *>(ws + L.samp_list);
    P.samp_count = reinterpret_cast<int *>(ws + L.samp_count);
    P.k0 = 0;
    P.k1 = K;
    P.gz = reinterpret_cast<const float *>(ws + L.gz);
    P.samp_t = reinterpret_cast<const char *>(crow);
    P.samp_d = reinterpret_cast<const char *>(shared ? crow + V : crow + (size_t)B * V);
    P.samp_stride = shared ? 2 : 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // 1. per-request set-up (lengths, greedy / sampled, the sampled-request count)
    sv::sv_prep<<<1, sv::prep_threads(P.B), 0, s>>>(P);
    // 2. the products of the target and draft rows; their epilogues leave the
    //    row statistics (and the logit at each draft token) in the workspace
    sv::LmStatsEpi ep{P.part, reinterpret_cast<float *>(ws + L.gz), draft_tokens, temperature,
                      P.npart, P.nslot, K, {K + 1, K}, {0, K + 1}, {0, K + 1}};
    sv::LmStatsEpi ed = ep;  // the draft rows as segment 0 of a launch of their own
    ed.rows_per_req[0] = K;
    ed.slot0[0] = K + 1;
    ed.tok_off[0] = K + 1;
    if (sv::g_prof_start) cudaEventRecord(sv::g_prof_start, s);
    if (shared) {
        if (sv::launch_lm_gemm(tHt, tHd, tWt, B * (K + 1), B * K, nullptr, 1, V, d, ep, dev_status,
                               *dv, s) != cudaSuccess)
            return SPEC_ERR_CUDA;
    } else if (sv::launch_lm_gemm(tHt, tHt, tWt, B * (K + 1), 0, nullptr, 1, V, d, ep, dev_status,
                                  *dv, s) != cudaSuccess ||
               sv::launch_lm_gemm(tHd, tHd, tWd, B * K, 0, nullptr, 1, V, d, ed, dev_status, *dv,
                                  s) != cudaSuccess) {
        return SPEC_ERR_CUDA;
    }
    if (sv::g_prof_end) cudaEventRecord(sv::g_prof_end, s);
    // 3. decisions; 4. the rows the sampled requests draw from, recomputed
    sv::launch_dependent(sv::decide_kernel<sv::kF32>(*dv, B), B, sv::kThreads, 0, s, P);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)B);
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, sv::lm_gather, P, static_cast<const uint16_t *>(hidden_target),
                               static_cast<const uint16_t *>(hidden_draft), d, hc,
                               shared ? hc + d : hc + (size_t)B * d, shared ? 2 : 1) != cudaSuccess)
            return SPEC_ERR_CUDA;
    }
    if (shared) {  // rows 2 li (target) and 2 li + 1 (draft), 2 * count of them
        sv::LmStoreEpi st{{crow, crow}};
        if (sv::launch_lm_gemm(tC0, tC0, tWt, 2 * B, 0, P.samp_count, 2, V, d, st, dev_status, *dv,
                               s) != cudaSuccess)
            return SPEC_ERR_CUDA;
    } else {
        sv::LmStoreEpi st{{crow, crow}}, sd{{crow + (size_t)B * V, crow + (size_t)B * V}};
        if (sv::launch_lm_gemm(tC0, tC0, tWt, B, 0, P.samp_count, 1, V, d, st, dev_status, *dv, s) !=
                cudaSuccess ||
            sv::launch_lm_gemm(tC1, tC1, tWd, B, 0, P.samp_count, 1, V, d, sd, dev_status, *dv, s) !=
                cudaSuccess)
            return SPEC_ERR_CUDA;
    }
    // 5. residual / bonus masses and the inverse CDF over the recomputed rows
    const bool vec = sv::vec_rows(V, SPEC_DTYPE_F32);
    long long g2 = (long long)dv->sms * dv->occ_sample[sv::kF32][vec ? 1 : 0];
    const long long g2_need = ((long long)B * P.nchunk + sv::kSWarps - 1) / sv::kSWarps;
    if (g2 > g2_need) g2 = g2_need;
    if (vec) {
        sv::launch_dependent(sv::sv_sample<sv::kF32, true>, (int)g2, sv::kSWarps * 32, sv::kSSmem, s, P);
        sv::launch_dependent(sv::sv_find<sv::kF32, true>, B,
                             sv::kFindWarps * 32, 0, s, P);
    } else {
        sv::launch_dependent(sv::sv_sample<sv::kF32, false>, (int)g2, sv::kSWarps * 32, 0, s, P);
        sv::launch_dependent(sv::sv_find<sv::kF32, false>, B,
                             sv::kFindWarps * 32, 0, s, P);
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

size_t spec_tree_workspace_bytes(int B, int N, int V, spec_dtype_t dtype) {
    if (N < 1 || N > SPEC_MAX_TREE || B < 1 || B >= (1 << 24) || V < 2 || V > SPEC_MAX_V) return 0;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
    return sv::layout(B, N - 1 > 0 ? N - 1 : 1, V, dtype).total;
}

spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t dtype,
                                      const int32_t *parent, const int32_t *node_tokens, int B,
                                      int N, int V, int32_t *out_tokens, int32_t *out_nodes,
                                      int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                      uint32_t *dev_status, void *stream) {
    if (N < 1 || N > SPEC_MAX_TREE || B < 1 || B >= (1 << 24) || V < 2 || V > SPEC_MAX_V)
        return SPEC_ERR_INVALID_ARG;
    const int K = N - 1 > 0 ? N - 1 : 1;  // the workspace layout of K = N - 1 holds N target rows
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    if (!sv::items_fit(B, K, V, dtype)) return SPEC_ERR_UNSUPPORTED;
    if (!target_logits || !parent || !node_tokens || !out_tokens || !out_nodes || !accept_len)
        return SPEC_ERR_INVALID_ARG;
    if ((uintptr_t)target_logits & 15u) return SPEC_ERR_INVALID_ARG;
    const sv::Layout L = sv::layout(B, K, V, dtype);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    sv::DevInfo *d = sv::dev_info();
    if (!d) return SPEC_ERR_CUDA;
    const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
    const bool vec = ((size_t)V * (size_t)esz) % 16u == 0;
    sv::Params P{};
    P.tgt = static_cast<const char *>(target_logits);
    P.drf = static_cast<const char *>(target_logits);  // no draft rows are listed
    P.B = B;
    P.K = N - 1;  // row n of the tree is target slot n
    P.V = V;
    P.nchunk = (int)sv::nchunk_for(V, dtype);
    P.npart = (int)sv::npart_for(V, dtype);
    P.nslot = 2 * K + 1;
    P.k0 = 0;
    P.k1 = P.K;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    char *ws = static_cast<char *>(workspace);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long rows = (long long)B * N;
    sv::sv_tree_rows<<<(unsigned)((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024), 256, 0, s>>>(P);
    const int g1 = d->sms * d->occ_p1[dtype == SPEC_DTYPE_BF16 ? sv::kBF16 : sv::kF32][vec ? 1 : 0];
    if (dtype == SPEC_DTYPE_BF16) {
        if (vec) sv::launch_dependent(sv::sv_pass1<sv::kBF16, true>, g1, sv::kP1Warps * 32, sv::kP1Smem, s, P);
        else sv::launch_dependent(sv::sv_pass1<sv::kBF16, false>, g1, sv::kP1Warps * 32, 0, s, P);
    } else {
        if (vec) sv::launch_dependent(sv::sv_pass1<sv::kF32, true>, g1, sv::kP1Warps * 32, sv::kP1Smem, s, P);
        else sv::launch_dependent(sv::sv_pass1<sv::kF32, false>, g1, sv::kP1Warps * 32, 0, s, P);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(sv::kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, sv::sv_tree_decide, P, parent, node_tokens, out_nodes);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

static spec_status_t verify_tree_impl(const void *target_logits, const void *draft_logits,
                                      spec_dtype_t dtype, const int32_t *parent,
                                      const int32_t *node_tokens, const float *temperature,
                                      uint64_t seed, int B, int N, int V, int32_t *out_tokens,
                                      int32_t *out_nodes, int32_t *accept_len, void *workspace,
                                      size_t workspace_bytes, uint32_t *dev_status, void *stream,
                                      int distinct) {
    if (N < 1 || N > SPEC_MAX_TREE || B < 1 || B >= (1 << 24) || V < 2 || V > SPEC_MAX_V)
        return SPEC_ERR_INVALID_ARG;
    const int K = N - 1 > 0 ? N - 1 : 1;  // the workspace layout of K = N - 1
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    if (!sv::items_fit(B, K, V, dtype)) return SPEC_ERR_UNSUPPORTED;
    if (!target_logits || (N > 1 && !draft_logits) || !parent || !node_tokens || !temperature ||
        !out_tokens || !out_nodes || !accept_len)
        return SPEC_ERR_INVALID_ARG;
    if (((uintptr_t)target_logits & 15u) || ((uintptr_t)draft_logits & 15u)) return SPEC_ERR_INVALID_ARG;
    const sv::Layout L = sv::layout(B, K, V, dtype);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    sv::DevInfo *d = sv::dev_info();
    if (!d) return SPEC_ERR_CUDA;
    const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
    const bool vec = ((size_t)V * (size_t)esz) % 16u == 0;
    sv::Params P{};
    P.tgt = static_cast<const char *>(target_logits);
    P.drf = static_cast<const char *>(N > 1 ? draft_logits : target_logits);
    P.temperature = temperature;
    P.seed = seed;
    P.B = B;
    P.K = N - 1;  // target slots 0..N-1 are the node rows, draft slots N..2N-2 the draft rows
    P.V = V;
    P.nchunk = (int)sv::nchunk_for(V, dtype);
    P.npart = (int)sv::npart_for(V, dtype);
    P.nslot = 2 * K + 1;
    P.k0 = 0;
    P.k1 = P.K;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    char *ws = static_cast<char *>(workspace);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    sv::sv_tree_rows_s<<<1, sv::kPrepThreads, 0, s>>>(P);
    const int g1 = d->sms * d->occ_p1[dtype == SPEC_DTYPE_BF16 ? sv::kBF16 : sv::kF32][vec ? 1 : 0];
    void (*walk)(sv::Params, const int32_t *, const int32_t *, int32_t *, int, int, int);
    if (dtype == SPEC_DTYPE_BF16) {
        if (vec) sv::launch_dependent(sv::sv_pass1<sv::kBF16, true>, g1, sv::kP1Warps * 32, sv::kP1Smem, s, P);
        else sv::launch_dependent(sv::sv_pass1<sv::kBF16, false>, g1, sv::kP1Warps * 32, 0, s, P);
        walk = vec ? sv::sv_tree_walk<sv::kBF16, true> : sv::sv_tree_walk<sv::kBF16, false>;
    } else {
        if (vec) sv::launch_dependent(sv::sv_pass1<sv::kF32, true>, g1, sv::kP1Warps * 32, sv::kP1Smem, s, P);
        else sv::launch_dependent(sv::sv_pass1<sv::kF32, false>, g1, sv::kP1Warps * 32, 0, s, P);
        walk = vec ? sv::sv_tree_walk<sv::kF32, true> : sv::sv_tree_walk<sv::kF32, false>;
    }
    // a cluster of cs CTAs (one per SM) per request while the batch leaves SMs free
    int cs = 1;
    while (cs < 8 && (long long)B * cs * 2 <= d->sms) cs *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * cs));
    cfg.blockDim = dim3(sv::kTreeThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // the slice of a node's two rows each CTA stages in shared memory, when it fits
    const long long nsteps = ((long long)V + sv::kTreeStep - 1) / sv::kTreeStep;
    const long long row_bytes = (nsteps + cs - 1) / cs * sv::kTreeStep * esz;
    const int stage = vec && 2 * row_bytes <= sv::kTreeStageMax ? (int)row_bytes : 0;
    // the attribute applies to the current device only: raised once per device
    bool &set = d->walk_smem[dtype == SPEC_DTYPE_BF16 ? 1 : 0][vec ? 1 : 0];
    if (!set) {
        if (cudaFuncSetAttribute(walk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sv::kTreeStageMax) != cudaSuccess)
            return SPEC_ERR_CUDA;
        set = true;
    }
    cfg.dynamicSmemBytes = stage ? (size_t)(2 * row_bytes) : 0;
    if (cudaLaunchKernelEx(&cfg, walk, P, parent, node_tokens, out_nodes, stage,
                           sv::g_diag_timeout ? 1 : 0, distinct) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_tree(const void *target_logits, const void *draft_logits,
                               spec_dtype_t dtype, const int32_t *parent,
                               const int32_t *node_tokens, const float *temperature, uint64_t seed,
                               int B, int N, int V, int32_t *out_tokens, int32_t *out_nodes,
                               int32_t *accept_len, void *workspace, size_t workspace_bytes,
                               uint32_t *dev_status, void *stream) {
    return verify_tree_impl(target_logits, draft_logits, dtype, parent, node_tokens, temperature,
                            seed, B, N, V, out_tokens, out_nodes, accept_len, workspace,
                            workspace_bytes, dev_status, stream, 0);
}

spec_status_t spec_verify_tree_distinct(const void *target_logits, const void *draft_logits,
                                        spec_dtype_t dtype, const int32_t *parent,
                                        const int32_t *node_tokens, const float *temperature,
                                        uint64_t seed, int B, int N, int V, int32_t *out_tokens,
                                        int32_t *out_nodes, int32_t *accept_len, void *workspace,
                                        size_t workspace_bytes, uint32_t *dev_status, void *stream) {
    return verify_tree_impl(target_logits, draft_logits, dtype, parent, node_tokens, temperature,
                            seed, B, N, V, out_tokens, out_nodes, accept_len, workspace,
                            workspace_bytes, dev_status, stream, 1);
}

spec_status_t spec_schedule_budget(const float *draft_maxprob, int B, int K, long long budget,
                                   int32_t *verify_len, void *stream) {
    if (B < 1 || B >= (1 << 24) || K < 1 || K > SPEC_MAX_K) return SPEC_ERR_INVALID_ARG;
    if (!draft_maxprob || !verify_len) return SPEC_ERR_INVALID_ARG;
    if ((long long)B * K > sv::kBudgetMaxN) return SPEC_ERR_UNSUPPORTED;
    sv::sv_schedule_budget<<<1, sv::kBudgetThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        draft_maxprob, B, K, budget, verify_len);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_schedule_len(const float *draft_maxprob, float threshold, int B, int K,
                                int32_t *verify_len, void *stream) {
    if (B < 1 || B >= (1 << 24) || K < 1 || K > SPEC_MAX_K) return SPEC_ERR_INVALID_ARG;
    if (!draft_maxprob || !verify_len) return SPEC_ERR_INVALID_ARG;
    const int nt = 256;
    sv::sv_schedule<<<(B + nt - 1) / nt, nt, 0, static_cast<cudaStream_t>(stream)>>>(
        draft_maxprob, threshold, B, K, verify_len);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ---------------------------------------------------------------- no-allocation entry
// Library-owned scratch for callers that cannot allocate (see the header).
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];
static void *g_noalloc_ptr[64];  // device address of the array, per device

spec_status_t spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                                  spec_dtype_t dtype, const int32_t *draft_tokens,
                                  const int32_t *verify_len, const float *temperature,
                                  uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                  int32_t *accept_len, uint32_t *dev_status, void *stream) {
    const size_t need = spec_verify_workspace_bytes(B, K, V, dtype);
    if (need == 0) {
        if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
        return SPEC_ERR_INVALID_ARG;
    }
    if (need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    if (!g_noalloc_ptr[dev]) {  // first call on this device: look up the array's address
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return SPEC_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    return sv::verify_impl(target_logits, draft_logits, dtype, draft_tokens, verify_len,
                           temperature, seed, B, K, V, out_tokens, accept_len,
                           g_noalloc_ptr[dev], (size_t)SPEC_NOALLOC_SCRATCH_BYTES, dev_status,
                           nullptr, nullptr, stream);
}

spec_status_t spec_verify_from_host(
    const void *target_host, const void *draft_host, spec_dtype_t dtype,
    const int32_t *draft_tokens_host, const int32_t *verify_len_host,
    const float *temperature_host, uint64_t seed, int B, int K, int V, void *target_dev,
    void *draft_dev, int32_t *draft_tokens_dev, int32_t *verify_len_dev, float *temperature_dev,
    int32_t *out_tokens_dev, int32_t *accept_len_dev, int32_t *out_tokens_host,
    int32_t *accept_len_host, void *workspace, size_t workspace_bytes, uint32_t *dev_status,
    void *stream, size_t *h2d_bytes) {
    if (!target_host || !draft_host || !draft_tokens_host || !temperature_host || !draft_tokens_dev ||
        !temperature_dev || !out_tokens_host || !accept_len_host || (verify_len_host && !verify_len_dev))
        return SPEC_ERR_INVALID_ARG;
    int32_t *vlen_dev = verify_len_host ? verify_len_dev : nullptr;
    // every argument check of the step first: nothing is copied on an error
    sv::Params P;
    sv::Layout L;
    const spec_status_t st = sv::step_params(P, target_dev, draft_dev, dtype, draft_tokens_dev,
                                             vlen_dev, temperature_dev, seed, B, K, V, out_tokens_dev,
                                             accept_len_dev, workspace, workspace_bytes, dev_status, L);
    if (st != SPEC_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t row = (size_t)V * (dtype == SPEC_DTYPE_BF16 ? 2u : 4u);
    sv::H2DRuns small, tgt, drf;
    small.s = tgt.s = drf.s = s;
    small.add(draft_tokens_host, draft_tokens_dev, (size_t)B * K * sizeof(int32_t));
    small.flush();
    if (verify_len_host) small.add(verify_len_host, verify_len_dev, (size_t)B * sizeof(int32_t));
    small.flush();
    small.add(temperature_host, temperature_dev, (size_t)B * sizeof(float));
    small.flush();
    const char *th = static_cast<const char *>(target_host), *dh = static_cast<const char *>(draft_host);
    char *td = static_cast<char *>(target_dev), *dd = static_cast<char *>(draft_dev);
    for (int b = 0; b < B; ++b) {
        // the rows request b's step reads (the rules of sv_prep)
        int Lb = verify_len_host ? verify_len_host[b] : K;
        Lb = Lb < 0 ? 0 : (Lb > K ? K : Lb);
        const float T = temperature_host[b];
        const bool greedy = !(std::isfinite(T) && T >= FLT_MIN);
        const size_t t0 = (size_t)b * (size_t)(K + 1) * row;
        tgt.add(th + t0, td + t0, (size_t)(Lb + 1) * row);
        if (!greedy) {
            const size_t d0 = (size_t)b * (size_t)K * row;
            drf.add(dh + d0, dd + d0, (size_t)Lb * row);
        }
    }
    tgt.flush();
    drf.flush();
    if (!small.ok || !tgt.ok || !drf.ok) return SPEC_ERR_CUDA;
    if (h2d_bytes) *h2d_bytes = small.total + tgt.total + drf.total;
    const spec_status_t sv_st = sv::verify_impl(target_dev, draft_dev, dtype, draft_tokens_dev, vlen_dev,
                                                temperature_dev, seed, B, K, V, out_tokens_dev,
                                                accept_len_dev, workspace, workspace_bytes, dev_status,
                                                nullptr, nullptr, stream);
    if (sv_st != SPEC_OK) return sv_st;
    if (cudaMemcpyAsync(out_tokens_host, out_tokens_dev, (size_t)B * (K + 1) * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(accept_len_host, accept_len_dev, (size_t)B * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

spec_status_t spec_verify_scheduled_from_host(
    const void *target_host, const void *draft_host, spec_dtype_t dtype,
    const int32_t *draft_tokens_host, const float *temperature_host,
    const float *draft_maxprob_host, uint64_t seed, int B, int K, int V, spec_sched_mode_t mode,
    float threshold, long long budget, void *target_dev, void *draft_dev,
    int32_t *draft_tokens_dev, float *temperature_dev, float *maxprob_dev, int32_t *verify_len_dev,
    int32_t *out_tokens_dev, int32_t *accept_len_dev, int32_t *out_tokens_host,
    int32_t *accept_len_host, int32_t *verify_len_host, void *workspace, size_t workspace_bytes,
    uint32_t *dev_status, void *stream, size_t *h2d_bytes) {
    if (mode != SPEC_SCHED_THRESHOLD && mode != SPEC_SCHED_BUDGET) return SPEC_ERR_INVALID_ARG;
    if (!draft_maxprob_host || !maxprob_dev || !verify_len_dev || !verify_len_host || !target_host ||
        !draft_host || !draft_tokens_host || !temperature_host || !draft_tokens_dev ||
        !temperature_dev || !out_tokens_host || !accept_len_host)
        return SPEC_ERR_INVALID_ARG;
    {  // every argument check of the step before the first copy
        sv::Params P;
        sv::Layout L;
        const spec_status_t st = sv::step_params(P, target_dev, draft_dev, dtype, draft_tokens_dev,
                                                 verify_len_dev, temperature_dev, seed, B, K, V,
                                                 out_tokens_dev, accept_len_dev, workspace,
                                                 workspace_bytes, dev_status, L);
        if (st != SPEC_OK) return st;
    }
    if (mode == SPEC_SCHED_BUDGET && (long long)B * K > sv::kBudgetMaxN) return SPEC_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t mp_bytes = (size_t)B * K * sizeof(float);
    if (cudaMemcpyAsync(maxprob_dev, draft_maxprob_host, mp_bytes, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    const spec_status_t ss = mode == SPEC_SCHED_THRESHOLD
                                 ? spec_schedule_len(maxprob_dev, threshold, B, K, verify_len_dev, stream)
                                 : spec_schedule_budget(maxprob_dev, B, K, budget, verify_len_dev, stream);
    if (ss != SPEC_OK) return ss;
    // the lengths decide which rows cross the host link: wait for them
    if (cudaMemcpyAsync(verify_len_host, verify_len_dev, (size_t)B * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    size_t n = 0;
    const spec_status_t st = spec_verify_from_host(
        target_host, draft_host, dtype, draft_tokens_host, verify_len_host, temperature_host, seed, B,
        K, V, target_dev, draft_dev, draft_tokens_dev, verify_len_dev, temperature_dev, out_tokens_dev,
        accept_len_dev, out_tokens_host, accept_len_host, workspace, workspace_bytes, dev_status,
        stream, &n);
    if (h2d_bytes) *h2d_bytes = n + mp_bytes;
    return st;
}

void spec_profile_events(void *ev_start, void *ev_end) {
    if (ev_start && ev_end) {
        sv::g_prof_start = static_cast<cudaEvent_t>(ev_start);
        sv::g_prof_end = static_cast<cudaEvent_t>(ev_end);
    } else {
        sv::g_prof_start = nullptr;
        sv::g_prof_end = nullptr;
    }
}

int spec_verify_kernel_count(void) { return sv::kKernelsPerVerify; }

spec_status_t spec_debug_force_wait_timeout(int enable) {
    sv::g_diag_timeout = enable != 0;
    return SPEC_OK;
}

const char *spec_status_str(spec_status_t status) {
    switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case SPEC_ERR_CUDA: return "CUDA launch failed";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

} // extern "C"
