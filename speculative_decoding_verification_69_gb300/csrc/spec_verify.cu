// spec_verify.cu -- sm_103a kernels and C ABI of the verification step.
//
// One call of spec_verify enqueues five kernels on the caller's stream:
//   1. sv_prep    per request: clamp the verify length, validate draft tokens,
//                 decide greedy / sampled, temperature scale; list the logit
//                 rows the step must read (target 0..L, draft 0..L-1 when
//                 sampled) -- all drafts are scored from one target pass and
//                 checked together ("speculative decoding от черновика до
//                 проверки" (braintools.ru), "Как это работает", steps 2-3).
//   2. sv_pass1   the logit stream: every needed row is read once, 4 KiB per
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
//                 chunk's vectors and elements.
// spec_schedule_len is one more small kernel (sv_schedule).
#include "spec_verify.h"
#include "sv_common.cuh"

#include <cuda_runtime.h>
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstdint>

namespace sv {

constexpr double kLog2E = 1.4426950408889634074;

struct ReqInfo {
    int L;        // effective verify length
    int greedy;   // 1: temperature 0 path
    float c;      // log2(e)/T rounded to float (statistics pass)
    float c_hi;   // two-float log2(e)/T, c_hi rounded toward zero (sampler)
    float c_lo;   // >= FLT_MIN
    float pad;
    double cd;    // log2(e)/T in double
    double inv_t; // 1/T in double
};

struct SampInfo {
    int mode;    // 0 none (greedy), 1 residual at row a, 2 bonus at row L
    int slot_t;  // target row slot to sample from
    int slot_d;  // draft row slot (mode 1)
    int a;       // emitted position
    float m_t;   // max logit of the target row
    float m_d;   // max logit of the draft row (mode 1)
    float rho_t; // 1/S of the target row (mode 1; 1 for the bonus)
    float rho_d; // 1/S of the draft row (mode 1)
    float c_hi, c_lo;
    int pad0, pad1;
    double u;    // sampling uniform
    double pad2;
};

struct Params {
    const char *tgt;
    const char *drf;
    const int32_t *tokens;
    const int32_t *verify_len;
    const float *temperature;
    unsigned long long seed;
    int B, K, V, nchunk, nslot;
    int32_t *out_tokens;
    int32_t *accept_len;
    uint32_t *dev_status;
    double *dbg_rows;  // [B, 2K+1, 2] or null
    double *dbg_probs; // [B, K, 2] or null
    // workspace
    ReqInfo *req;
    int *row_count;
    int4 *rows;        // (b, slot, greedy, log2(e)/T float bits) of every needed row, request-major
    float4 *part;      // [B, nslot, nchunk]: statistics-pass partials
    SampInfo *samp;    // [B]
    float4 *sub;       // [B, nchunk]: sampler chunk masses A, B, W
    float4 *sexact;    // [B, nchunk]: exact sums of e (hi, lo) and e' (hi, lo)
};

__device__ __forceinline__ const char *row_ptr(const Params &P, int b, int slot, int esz) {
    if (slot <= P.K)
        return P.tgt + ((size_t)b * (size_t)(P.K + 1) + (size_t)slot) * (size_t)P.V * esz;
    return P.drf + ((size_t)b * (size_t)P.K + (size_t)(slot - P.K - 1)) * (size_t)P.V * esz;
}

__device__ __forceinline__ float load_logit(const char *row, int dt, int x) {
    if (dt == kBF16) {
        uint16_t h = __ldg(reinterpret_cast<const uint16_t *>(row) + x);
        return __uint_as_float((uint32_t)h << 16);
    }
    return __ldg(reinterpret_cast<const float *>(row) + x);
}

// ------------------------------------------------------------------ 1. prep

constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) sv_prep(Params P) {
    __shared__ int warp_tot[kPrepThreads / 32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < P.B; base += kPrepThreads) {
        const int b = base + tid;
        int n = 0, L = 0, greedy = 1;
        float cval = 0.f;
        if (b < P.B) {
            uint32_t st = 0;
            L = P.verify_len ? P.verify_len[b] : P.K;
            if (L < 0) { L = 0; st |= SPEC_DEV_BAD_LEN; }
            if (L > P.K) { L = P.K; st |= SPEC_DEV_BAD_LEN; }
            for (int k = 0; k < L; ++k) {
                int x = P.tokens[(size_t)b * P.K + k];
                if (x < 0 || x >= P.V) { L = k; st |= SPEC_DEV_BAD_TOKEN; break; }
            }
            const float T = P.temperature[b];
            greedy = !(isfinite(T) && T >= FLT_MIN);
            ReqInfo ri;
            ri.L = L;
            ri.greedy = greedy;
            if (!greedy) {
                double c = kLog2E / (double)T;
                float chi = __double2float_rz(c);
                float clo = __double2float_rn(c - (double)chi);
                if (!(clo >= FLT_MIN)) clo = FLT_MIN;
                ri.c = __double2float_rn(c);
                ri.c_hi = chi;
                ri.c_lo = clo;
                ri.cd = c;
                ri.inv_t = 1.0 / (double)T;
            } else {
                ri.c = 0.f; ri.c_hi = 0.f; ri.c_lo = 0.f; ri.cd = 0.0; ri.inv_t = 0.0;
            }
            ri.pad = 0.f;
            P.req[b] = ri;
            cval = ri.c;
            if (st && P.dev_status) atomicOr(P.dev_status, st);
            n = L + 1 + (greedy ? 0 : L);
        }
        // block exclusive scan of n
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_tot[w] = incl;
        __syncthreads();
        int woff = 0;
        for (int i = 0; i < w; ++i) woff += warp_tot[i];
        int block_tot = 0;
        for (int i = 0; i < kPrepThreads / 32; ++i) block_tot += warp_tot[i];
        const int off = carry_s + woff + incl - n;
        if (b < P.B) {
            for (int r = 0; r < n; ++r) {
                int slot = r <= L ? r : (P.K + 1 + (r - L - 1));
                P.rows[off + r] = make_int4(b, slot, greedy, __float_as_int(cval));
            }
        }
        __syncthreads();
        if (tid == 0) carry_s += block_tot;
        __syncthreads();
    }
    if (tid == 0) *P.row_count = carry_s;
}

// ------------------------------------------------------------------ 2. statistics pass

constexpr int kP1Warps = 8;  // warps per CTA; every warp runs its own copy pipeline
constexpr int kStages = 3;   // bulk-copy stages per warp
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded wait: 2 s

struct P1Shared {
    uint4 buf[kP1Warps][kStages][kChunkBytes / 16];
    unsigned long long bar[kP1Warps][kStages];
};

__device__ __forceinline__ void p1_issue(const Params &P, uint32_t item, uint4 *dst,
                                         unsigned long long *bar, int esz) {
    const uint32_t ri = item / (uint32_t)P.nchunk;
    const uint32_t c = item - ri * (uint32_t)P.nchunk;
    const int4 bs = P.rows[ri];
    const char *row = row_ptr(P, bs.x, bs.y, esz);
    const uint32_t ce = kChunkBytes / esz;
    const uint32_t e0 = c * ce;
    const uint32_t n = min(ce, (uint32_t)P.V - e0);
    const uint32_t bytes = n * (uint32_t)esz;
    mbar_expect_tx(reinterpret_cast<uint64_t *>(bar), bytes);
    bulk_g2s(dst, row + (size_t)e0 * esz, bytes, reinterpret_cast<uint64_t *>(bar));
}

// One item = 4 KiB of one needed logit row.  Warps are independent: each keeps
// kStages bulk copies in flight into its own shared-memory ring, reads a stage
// into registers, and writes one partial per item:
//   greedy rows:  { m_c = max z, -, -, lowest index of m_c }
//   sampled rows: { m_c = max z, s_c = sum 2^((z - m_c) c), -, -1 }
template <int DT, bool VEC>
__global__ void __launch_bounds__(kP1Warps * 32) sv_pass1(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = chunk_elems<DT>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    P1Shared &sh = *reinterpret_cast<P1Shared *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t nitems = (uint32_t)(*P.row_count) * (uint32_t)P.nchunk;
    const uint32_t first = blockIdx.x * kP1Warps + warp;
    const uint32_t stride = gridDim.x * kP1Warps;
    uint4(*buf)[kChunkBytes / 16] = sh.buf[warp];
    unsigned long long *bar = sh.bar[warp];
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const uint4 neg_inf = make_uint4(ni, ni, ni, ni);
    if (VEC) {
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(reinterpret_cast<uint64_t *>(&bar[s]), 1);
            fence_mbar_init();
            for (int s = 0; s < kStages; ++s) {
                const uint32_t it = first + (uint32_t)s * stride;
                if (it < nitems) p1_issue(P, it, buf[s], &bar[s], ESZ);
            }
        }
        __syncwarp();
    }
    uint32_t k = 0;
    bool failed = false;
    for (uint32_t item = first; item < nitems; item += stride, ++k) {
        const int s = (int)(k % kStages);
        const uint32_t par = (k / kStages) & 1u;
        const uint32_t ri = item / (uint32_t)P.nchunk;
        const uint32_t c = item - ri * (uint32_t)P.nchunk;
        const int4 bs = P.rows[ri];
        const int b = bs.x, slot = bs.y;
        const uint32_t e0 = c * CE;
        const int nvec = (int)((min((uint32_t)CE, (uint32_t)P.V - e0) + EPV - 1) / EPV);
        uint4 v[kVecPerLane];
        if (VEC) {
            if (!mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[s]), par, kWaitLimitNs)) {
                failed = true;
                break;
            }
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i) {
                const int q = i * 32 + lane;
                v[i] = q < nvec ? buf[s][q] : neg_inf;
            }
            __syncwarp();
            if (lane == 0) {
                const uint32_t nx = item + (uint32_t)kStages * stride;
                if (nx < nitems) {
                    fence_proxy_async();
                    p1_issue(P, nx, buf[s], &bar[s], ESZ);
                }
            }
        } else {
            const char *row = row_ptr(P, b, slot, ESZ);
#pragma unroll
            for (int i = 0; i < kVecPerLane; ++i)
                v[i] = load_vec<DT, false>(row, (long long)e0 + (long long)(i * 32 + lane) * EPV, P.V);
        }
        const ReqInfo rq = P.req[b];
        float lm = -INFINITY;
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) lm = fmaxf(lm, vec_max<DT>(v[i]));
        const float m = warp_max(lm);
        float4 out;
        if (rq.greedy) {
            int idx = INT_MAX;
            if (lm == m) {
#pragma unroll
                for (int i = 0; i < kVecPerLane; ++i)
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (idx == INT_MAX && elem<DT>(v[i], e) == m)
                            idx = (int)e0 + (i * 32 + lane) * EPV + e;
            }
            idx = warp_min_int(idx);
            out = make_float4(m, 0.f, 0.f, __int_as_float(idx));
        } else {
            float ssum = 0.f;
            if (m > -INFINITY) {
                const float2 m2 = make_float2(m, m), c2 = make_float2(rq.c, rq.c);
                float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kVecPerLane; ++i) {
#pragma unroll
                    for (int e = 0; e < EPV; e += 4) {
                        const float2 t0 = mul2(sub2(make_float2(elem<DT>(v[i], e), elem<DT>(v[i], e + 1)), m2), c2);
                        a0 = add2(a0, make_float2(ex2(t0.x), ex2(t0.y)));
                        const float2 t1 = mul2(sub2(make_float2(elem<DT>(v[i], e + 2), elem<DT>(v[i], e + 3)), m2), c2);
                        a1 = add2(a1, make_float2(ex2(t1.x), ex2(t1.y)));
                    }
                }
                const float2 a = add2(a0, a1);
                ssum = a.x + a.y;
            }
            ssum = warp_sum(ssum);
            out = make_float4(m, ssum, 0.f, __int_as_float(-1));
        }
        if (lane == 0) P.part[((size_t)b * P.nslot + slot) * P.nchunk + c] = out;
    }
    if (VEC && failed) {
        // report, then let every copy this warp still has in flight land
        if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        for (uint32_t kk = k; kk < k + kStages; ++kk) {
            if (first + kk * stride >= nitems) break;
            mbar_wait_bounded(reinterpret_cast<uint64_t *>(&bar[kk % kStages]), (kk / kStages) & 1u,
                              kWaitLimitNs);
        }
    }
}

// ------------------------------------------------------------------ 3. decide

template <int DT>
__global__ void __launch_bounds__(kThreads) sv_decide(Params P) {
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = P.K;
    const ReqInfo rq = P.req[b];
    const int L = rq.L;
    const bool greedy = rq.greedy != 0;
    __shared__ float s_m[2 * SPEC_MAX_K + 1];
    __shared__ float s_S[2 * SPEC_MAX_K + 1];
    __shared__ int s_amax[SPEC_MAX_K + 1];
    __shared__ int s_a;
    const int nrows = greedy ? L + 1 : 2 * L + 1;
    // row statistics: one warp per row, lanes over the row's chunk partials
    for (int r = warp; r < nrows; r += kWarps) {
        const int slot = r <= L ? r : K + 1 + (r - L - 1);
        const float4 *pp = P.part + ((size_t)b * P.nslot + slot) * P.nchunk;
        float m = -INFINITY;
        for (int c = lane; c < P.nchunk; c += 32) m = fmaxf(m, pp[c].x);
        m = warp_max(m);
        float S = 0.f;
        int amax = INT_MAX;
        if (greedy) {
            for (int c = lane; c < P.nchunk; c += 32) {
                const float4 q = pp[c];
                if (q.x == m) amax = min(amax, __float_as_int(q.w));
            }
            amax = warp_min_int(amax);
        } else if (m > -INFINITY) {
            for (int c = lane; c < P.nchunk; c += 32) {
                const float4 q = pp[c];
                if (q.x > -INFINITY) S += q.y * ex2((q.x - m) * rq.c);
            }
            S = warp_sum(S);
        }
        if (lane == 0) {
            s_m[slot] = m;
            s_S[slot] = S;
            if (slot <= K) s_amax[slot] = amax;
        }
    }
    __syncthreads();
    if (warp == 0) {
        bool acc = true;
        if (lane < L) {
            const int x = P.tokens[(size_t)b * K + lane];
            if (greedy) {
                acc = (x == s_amax[lane]);
            } else {
                const float g = load_logit(row_ptr(P, b, lane, Fmt<DT>::kESZ), DT, x);
                const float gd = load_logit(row_ptr(P, b, K + 1 + lane, Fmt<DT>::kESZ), DT, x);
                const float St = s_S[lane], Sd = s_S[K + 1 + lane];
                const double p = St > 0.f ? exp2(((double)g - (double)s_m[lane]) * rq.cd) / (double)St : 0.0;
                const double q = Sd > 0.f ? exp2(((double)gd - (double)s_m[K + 1 + lane]) * rq.cd) / (double)Sd : 0.0;
                const double u = uniform_accept(P.seed, (uint32_t)b, (uint32_t)lane);
                acc = u * q < p;
                if (P.dbg_probs) {
                    P.dbg_probs[((size_t)b * K + lane) * 2 + 0] = p;
                    P.dbg_probs[((size_t)b * K + lane) * 2 + 1] = q;
                }
            }
        }
        const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc);
        const int a = rej ? min(__ffs(rej) - 1, L) : L;
        if (lane == 0) s_a = a;
    }
    __syncthreads();
    const int a = s_a;
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    for (int k = tid; k <= K; k += kThreads) {
        int v = -1;
        if (k < a) v = P.tokens[(size_t)b * K + k];
        else if (k == a && greedy) v = s_amax[a];
        out[k] = v;
    }
    if (tid == 0) {
        P.accept_len[b] = a;
        SampInfo si;
        si.mode = greedy ? 0 : (a < L ? 1 : 2);
        si.a = a;
        si.slot_t = a;
        si.slot_d = K + 1 + a;
        si.m_t = s_m[a];
        si.rho_t = 1.f;
        si.m_d = 0.f;
        si.rho_d = 0.f;
        if (si.mode == 1) {
            si.rho_t = 1.f / s_S[a];
            si.m_d = s_m[K + 1 + a];
            si.rho_d = 1.f / s_S[K + 1 + a];
        }
        si.c_hi = rq.c_hi;
        si.c_lo = rq.c_lo;
        si.u = greedy ? 0.0 : uniform_sample(P.seed, (uint32_t)b, (uint32_t)a);
        P.samp[b] = si;
    }
    if (P.dbg_rows) {
        const int nslot = 2 * K + 1;
        for (int sl = tid; sl < nslot; sl += kThreads) {
            double m = NAN, ls = NAN;
            const bool read = !greedy && (sl <= L || (sl >= K + 1 && sl - K - 1 < L));
            if (read) {
                m = (double)s_m[sl] * rq.inv_t;
                ls = log((double)s_S[sl]);
            }
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 0] = m;
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 1] = ls;
        }
        if (P.dbg_probs)
            for (int k = (greedy ? 0 : L) + tid; k < K; k += kThreads) {
                P.dbg_probs[((size_t)b * K + k) * 2 + 0] = NAN;
                P.dbg_probs[((size_t)b * K + k) * 2 + 1] = NAN;
            }
    }
}

// ------------------------------------------------------------------ 4. sampler pass

// Per element pair (target z, draft z') of the sampled row (pair):
//   e = 2^((z - m) c), e' = 2^((z' - m') c) with the row maxima and two-float c;
//   a = e * rho, b = e' * rho' with rho = 1/S from the statistics pass.
// Per chunk: A = sum of a over {a > b}, B = sum of b over {a > b}, W = sum of a,
// and the exact sums of e and e'.  The residual mass of a chunk is then
// kappa A - kappa' B with kappa = 1 / (rho * sum e) (exact normaliser).
template <int DT>
__device__ __forceinline__ void pair_weights(float zt, float zd, float2 m2, float2 chi2,
                                             float2 clo2, float2 rho2, float2 &ee, float2 &ab) {
    ee = weight2(make_float2(zt, zd), m2, chi2, clo2);
    ab = mul2(ee, rho2);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sv_sample(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = chunk_elems<DT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t nitems = (uint32_t)P.B * (uint32_t)P.nchunk;
    const uint32_t stride = gridDim.x * kWarps;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    for (uint32_t item = blockIdx.x * kWarps + warp; item < nitems; item += stride) {
        const uint32_t b = item / (uint32_t)P.nchunk;
        const uint32_t c = item - b * (uint32_t)P.nchunk;
        const SampInfo si = P.samp[b];
        if (si.mode == 0) continue;
        const bool resid = si.mode == 1;
        const char *rowt = row_ptr(P, (int)b, si.slot_t, ESZ);
        const char *rowd = resid ? row_ptr(P, (int)b, si.slot_d, ESZ) : rowt;
        const long long e0 = (long long)c * CE;
        uint4 vt[kVecPerLane], vd[kVecPerLane];
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
            const long long q = e0 + (long long)(i * 32 + lane) * EPV;
            vt[i] = load_vec<DT, VEC>(rowt, q, P.V);
            vd[i] = resid ? load_vec<DT, VEC>(rowd, q, P.V) : make_uint4(ni, ni, ni, ni);
        }
        const float2 m2 = make_float2(si.m_t, si.m_d);
        const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
        const float2 rho2 = make_float2(si.rho_t, si.rho_d);
        BiasAcc2 acc;
        acc.init(1.0f);
        float A = 0.f, Bs = 0.f, W = 0.f;
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                float2 ee, ab;
                pair_weights<DT>(elem<DT>(vt[i], e), elem<DT>(vd[i], e), m2, chi2, clo2, rho2, ee, ab);
                acc.add(ee);
                W = __fadd_rn(W, ab.x);
                if (ab.x > ab.y) {
                    A = __fadd_rn(A, ab.x);
                    Bs = __fadd_rn(Bs, ab.y);
                }
            }
        }
        A = warp_sum(A);
        Bs = warp_sum(Bs);
        W = warp_sum(W);
        FF st = warp_sum_ff(ff_add(FF{__fsub_rn(acc.h.x, 1.0f), acc.l.x}, FF{0.f, 0.f}));
        FF sd = warp_sum_ff(ff_add(FF{__fsub_rn(acc.h.y, 1.0f), acc.l.y}, FF{0.f, 0.f}));
        if (lane == 0) {
            P.sub[(size_t)b * P.nchunk + c] = make_float4(A, Bs, W, 0.f);
            P.sexact[(size_t)b * P.nchunk + c] = make_float4(st.hi, st.lo, sd.hi, sd.lo);
        }
    }
}

// ------------------------------------------------------------------ 5. inverse CDF

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sv_find(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = chunk_elems<DT>();
    __shared__ double red_d[kWarps];
    __shared__ double s_tot[4];
    __shared__ int s_chunk;
    __shared__ double s_base;
    __shared__ int s_tok;
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const SampInfo si = P.samp[b];
    if (si.mode == 0) return;
    const bool resid = si.mode == 1;
    const int nch = P.nchunk;
    const float4 *sub = P.sub + (size_t)b * nch;
    const float4 *sex = P.sexact + (size_t)b * nch;
    // exact normalisers and residual / target masses
    double st = 0.0, sd = 0.0, zr = 0.0, zw = 0.0;
    for (int c = tid; c < nch; c += kThreads) {
        const float4 e = sex[c];
        st += (double)e.x + (double)e.y;
        sd += (double)e.z + (double)e.w;
    }
    st = warp_sum_d(st);
    sd = warp_sum_d(sd);
    if (lane == 0) { red_d[warp] = st; }
    __syncthreads();
    if (tid == 0) { double t = 0; for (int i = 0; i < kWarps; ++i) t += red_d[i]; s_tot[0] = t; }
    __syncthreads();
    if (lane == 0) { red_d[warp] = sd; }
    __syncthreads();
    if (tid == 0) { double t = 0; for (int i = 0; i < kWarps; ++i) t += red_d[i]; s_tot[1] = t; }
    __syncthreads();
    const double kt = resid ? 1.0 / ((double)si.rho_t * s_tot[0]) : 1.0;
    const double kd = resid ? 1.0 / ((double)si.rho_d * s_tot[1]) : 0.0;
    // chunk masses: contiguous blocks of chunks per thread
    const int per = (nch + kThreads - 1) / kThreads;
    const int c0 = tid * per, c1 = min(nch, c0 + per);
    for (int c = c0; c < c1; ++c) {
        const float4 q = sub[c];
        zr += resid ? fmax(0.0, kt * (double)q.x - kd * (double)q.y) : (double)q.z;
        zw += (double)q.z;
    }
    // totals
    double tr = warp_sum_d(zr), tw = warp_sum_d(zw);
    __syncthreads();
    if (lane == 0) red_d[warp] = tr;
    __syncthreads();
    if (tid == 0) { double t = 0; for (int i = 0; i < kWarps; ++i) t += red_d[i]; s_tot[2] = t; }
    __syncthreads();
    if (lane == 0) red_d[warp] = tw;
    __syncthreads();
    if (tid == 0) { double t = 0; for (int i = 0; i < kWarps; ++i) t += red_d[i]; s_tot[3] = t; s_chunk = INT_MAX; s_tok = INT_MAX; }
    __syncthreads();
    const bool use_w = !resid || !(s_tot[2] > 0.0);  // bonus, or residual with zero mass
    const double Z = use_w ? s_tot[3] : s_tot[2];
    const double theta = si.u * Z;
    // exclusive prefix of this thread's block
    const double mine = use_w ? zw : zr;
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();
    if (lane == 31) red_d[warp] = incl;
    __syncthreads();
    double off = 0.0;
    for (int i = 0; i < warp; ++i) off += red_d[i];
    double base = off + incl - mine;
    int my_c = INT_MAX;
    double my_base = 0.0;
    if (base <= theta && base + mine > theta) {
        for (int c = c0; c < c1; ++c) {
            const float4 q = sub[c];
            const double v = use_w ? (double)q.z : (resid ? fmax(0.0, kt * (double)q.x - kd * (double)q.y) : (double)q.z);
            if (base + v > theta) {
                my_c = c;
                my_base = base;
                break;
            }
            base += v;
        }
        if (my_c != INT_MAX) atomicMin(&s_chunk, my_c);
    }
    __syncthreads();
    if (my_c != INT_MAX && my_c == s_chunk) s_base = my_base;
    __syncthreads();
    int ch = s_chunk;
    double th_local;
    if (ch == INT_MAX) {
        // rounding left no crossing: the last chunk with positive mass
        ch = nch - 1;
        for (int c = nch - 1; c >= 0; --c) {
            const float4 q = sub[c];
            const double v = use_w ? (double)q.z : fmax(0.0, kt * (double)q.x - kd * (double)q.y);
            if (v > 0.0) { ch = c; break; }
        }
        th_local = INFINITY;
    } else {
        th_local = theta - s_base;
    }
    if (warp == 0) {
        const char *rowt = row_ptr(P, b, si.slot_t, ESZ);
        const char *rowd = resid ? row_ptr(P, b, si.slot_d, ESZ) : rowt;
        const long long e0 = (long long)ch * CE;
        const uint32_t ni = Fmt<DT>::kNegInfWord;
        const float2 m2 = make_float2(si.m_t, si.m_d);
        const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
        const float2 rho2 = make_float2(si.rho_t, si.rho_d);
        const float dkt = (float)(kt - 1.0), dkd = (float)(kd - 1.0);
        double run = 0.0;
        int found = INT_MAX, last_pos = -1;
        for (int i = 0; i < kVecPerLane && found == INT_MAX; ++i) {
            const long long q0 = e0 + (long long)(i * 32 + lane) * EPV;
            const uint4 vt = load_vec<DT, VEC>(rowt, q0, P.V);
            const uint4 vd = (resid && !use_w) ? load_vec<DT, VEC>(rowd, q0, P.V) : make_uint4(ni, ni, ni, ni);
            float w[EPV];
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                float2 ee, ab;
                pair_weights<DT>(elem<DT>(vt, e), elem<DT>(vd, e), m2, chi2, clo2,
                                 (resid && !use_w) ? rho2 : make_float2(si.rho_t, 0.f), ee, ab);
                float wv;
                if (use_w) wv = ab.x;
                else wv = ab.x > ab.y ? fmaxf(__fsub_rn(__fmaf_rn(ab.x, dkt, ab.x), __fmaf_rn(ab.y, dkd, ab.y)), 0.f) : 0.f;
                w[e] = wv;
                if (wv > 0.f && q0 + e < P.V) last_pos = (int)(q0 + e);
            }
            float vs = w[0];
#pragma unroll
            for (int e = 1; e < EPV; ++e) vs = __fadd_rn(vs, w[e]);
            float inc = vs;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc = __fadd_rn(inc, u);
            }
            const double lo_edge = run + (double)(inc - vs);
            int tok = INT_MAX;
            if (lo_edge <= th_local && lo_edge + (double)vs > th_local) {
                float ps = 0.f;
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    ps = e == 0 ? w[0] : __fadd_rn(ps, w[e]);
                    if (tok == INT_MAX && lo_edge + (double)ps > th_local) tok = (int)(q0 + e);
                }
            }
            found = warp_min_int(tok);
            run += (double)__shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        if (found == INT_MAX) {
            int lp = last_pos;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xFFFFFFFFu, lp, o));
            found = lp >= 0 ? lp : (int)e0;
        }
        if (lane == 0) P.out_tokens[(size_t)b * (P.K + 1) + si.a] = found;
    }
}

// ------------------------------------------------------------------ schedule

__global__ void sv_schedule(const float *__restrict__ mp, float thr, int B, int K,
                            int32_t *__restrict__ out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    float prod = 1.0f;
    int L = 0;
    for (int k = 0; k < K; ++k) {
        prod = __fmul_rn(prod, mp[(size_t)b * K + k]);
        if (prod >= thr) L = k + 1;
        else break;
    }
    out[b] = L;
}

// ------------------------------------------------------------------ host side

struct Layout {
    size_t req, row_count, rows, part, samp, sub, sexact, total;
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
    L.part = off; off = align256(off + sizeof(float4) * (size_t)B * nslot * nchunk);
    L.samp = off; off = align256(off + sizeof(SampInfo) * (size_t)B);
    L.sub = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.sexact = off; off = align256(off + sizeof(float4) * (size_t)B * nchunk);
    L.total = off;
    return L;
}

struct DevInfo {
    int sms = 0;
    int occ_p1[2][2] = {{0, 0}, {0, 0}};
    int occ_sample[2][2] = {{0, 0}, {0, 0}};
    bool ok = false;
};

static DevInfo g_dev[64];
constexpr size_t kP1Smem = sizeof(P1Shared);

template <int DT, bool VEC>
static bool setup_kernels(DevInfo &d) {
    const size_t smem = VEC ? kP1Smem : 0;
    if (VEC && cudaFuncSetAttribute(sv_pass1<DT, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem) != cudaSuccess)
        return false;
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_pass1<DT, VEC>, kP1Warps * 32, smem) !=
        cudaSuccess)
        return false;
    d.occ_p1[DT][VEC] = o > 0 ? o : 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_sample<DT, VEC>, kThreads, 0) !=
        cudaSuccess)
        return false;
    d.occ_sample[DT][VEC] = o > 0 ? o : 1;
    return true;
}

static const DevInfo *dev_info() {
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

template <int DT, bool VEC>
static void launch_all(const Params &P, const DevInfo &d, cudaStream_t s) {
    sv_prep<<<1, kPrepThreads, 0, s>>>(P);
    const int g1 = d.sms * d.occ_p1[DT][VEC];
    if (g_prof_start) cudaEventRecord(g_prof_start, s);
    sv_pass1<DT, VEC><<<g1, kP1Warps * 32, VEC ? kP1Smem : 0, s>>>(P);
    if (g_prof_end) cudaEventRecord(g_prof_end, s);
    sv_decide<DT><<<P.B, kThreads, 0, s>>>(P);
    const long long warps_needed = (long long)P.B * P.nchunk;
    long long g2 = (long long)d.sms * d.occ_sample[DT][VEC];
    const long long g2_need = (warps_needed + kWarps - 1) / kWarps;
    if (g2 > g2_need) g2 = g2_need;
    sv_sample<DT, VEC><<<(int)g2, kThreads, 0, s>>>(P);
    sv_find<DT, VEC><<<P.B, kThreads, 0, s>>>(P);
}

static spec_status_t verify_impl(const void *target_logits, const void *draft_logits,
                                 spec_dtype_t dtype, const int32_t *draft_tokens,
                                 const int32_t *verify_len, const float *temperature,
                                 uint64_t seed, int B, int K, int V, int32_t *out_tokens,
                                 int32_t *accept_len, void *workspace, size_t workspace_bytes,
                                 uint32_t *dev_status, double *row_stats, double *probs,
                                 void *stream) {
    if (!sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    if (!items_fit(B, K, V, dtype)) return SPEC_ERR_UNSUPPORTED;
    if (!target_logits || !draft_logits || !draft_tokens || !temperature || !out_tokens ||
        !accept_len)
        return SPEC_ERR_INVALID_ARG;
    if (((uintptr_t)target_logits & 15u) || ((uintptr_t)draft_logits & 15u))
        return SPEC_ERR_INVALID_ARG;
    const Layout L = layout(B, K, V, dtype);
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u))
        return SPEC_ERR_WORKSPACE;
    const DevInfo *d = dev_info();
    if (!d) return SPEC_ERR_CUDA;
    const int esz = dtype == SPEC_DTYPE_BF16 ? 2 : 4;
    const bool vec = ((size_t)V * (size_t)esz) % 16u == 0;
    Params P{};
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
    P.nslot = 2 * K + 1;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    P.dbg_rows = row_stats;
    P.dbg_probs = probs;
    char *ws = static_cast<char *>(workspace);
    P.req = reinterpret_cast<ReqInfo *>(ws + L.req);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int4 *>(ws + L.rows);
    P.part = reinterpret_cast<float4 *>(ws + L.part);
    P.samp = reinterpret_cast<SampInfo *>(ws + L.samp);
    P.sub = reinterpret_cast<float4 *>(ws + L.sub);
    P.sexact = reinterpret_cast<float4 *>(ws + L.sexact);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_DTYPE_BF16) {
        if (vec) launch_all<kBF16, true>(P, *d, s);
        else launch_all<kBF16, false>(P, *d, s);
    } else {
        if (vec) launch_all<kF32, true>(P, *d, s);
        else launch_all<kF32, false>(P, *d, s);
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

} // namespace sv

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
