// spec_verify.cu -- sm_103a kernels and C ABI of the verification step.
//
// One call of spec_verify enqueues five kernels on the caller's stream:
//   1. sv_prep       per request: clamp the verify length, validate draft tokens,
//                    decide greedy / sampled, temperature scale; list the logit
//                    rows the step must read (target 0..L, draft 0..L-1 when
//                    sampled) -- the parallel formulation of the check in
//                    "speculative decoding от черновика до проверки"
//                    (braintools.ru), "Как это работает", steps 2-3.
//   2. sv_rowstats   persistent over (row, tile): streams every needed logit
//                    once with 128-bit loads; per tile the exact max, and
//                    either the lowest-index argmax (greedy) or the sum of
//                    2^((z - m_t) log2(e)/T) (sampled).
//   3. sv_decide     per request: combines tiles into row statistics, draws the
//                    Philox uniforms, applies the acceptance rule of
//                    "Спекулятивный декодинг в проде" (kiosknews.app),
//                    "Немного теории", "Правило проверки" (or the argmax
//                    comparison for temperature 0), finds the first rejection
//                    with a warp ballot, writes the accepted prefix, and
//                    prepares the residual / bonus sampler.
//   4. sv_sampletile per (request, tile) of the one row (pair) to sample from:
//                    tile masses of max(0, p - q) (rejection) and of p.
//   5. sv_find       per request: inverse CDF over tiles, then inside the
//                    chosen tile over 16-byte vectors and elements.
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
    float c_hi;   // two-float log2(e)/T, c_hi rounded toward zero
    float c_lo;   // >= FLT_MIN
    double c;     // log2(e)/T in double
    double inv_t; // 1/T in double
};

struct SampInfo {
    int mode;   // 0 none (greedy), 1 residual at row a, 2 bonus at row L
    int slot_t; // target row slot to sample from
    int slot_d; // draft row slot (mode 1)
    int a;      // emitted position
    double u;   // sampling uniform
};

struct Params {
    const char *tgt;
    const char *drf;
    const int32_t *tokens;
    const int32_t *verify_len;
    const float *temperature;
    unsigned long long seed;
    int B, K, V, ntile, nslot;
    int32_t *out_tokens;
    int32_t *accept_len;
    uint32_t *dev_status;
    double *dbg_rows;  // [B, 2K+1, 2] or null
    double *dbg_probs; // [B, K, 2] or null
    // workspace
    ReqInfo *req;
    int *row_count;
    int2 *rows;        // (b, slot)
    float4 *stats;     // [B, nslot, ntile]: m, S_hi, S_lo, argmax bits
    SampInfo *samp;    // [B]
    float4 *alpha;     // [B, ntile]: target (hi, lo), draft (hi, lo)
    float4 *ztile;     // [B, ntile]: residual (hi, lo), p (hi, lo)
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
                ri.c_hi = chi;
                ri.c_lo = clo;
                ri.c = c;
                ri.inv_t = 1.0 / (double)T;
            } else {
                ri.c_hi = 0.f; ri.c_lo = 0.f; ri.c = 0.0; ri.inv_t = 0.0;
            }
            P.req[b] = ri;
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
                P.rows[off + r] = make_int2(b, slot);
            }
        }
        __syncthreads();
        if (tid == 0) carry_s += block_tot;
        __syncthreads();
    }
    if (tid == 0) *P.row_count = carry_s;
}

// ------------------------------------------------------------------ 2. row stats

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sv_rowstats(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int TE = tile_elems<DT>();
    __shared__ float red_f[2 * kWarps];
    __shared__ int red_i[kWarps];
    const int tid = threadIdx.x;
    const long long total = (long long)(*P.row_count) * P.ntile;
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const int ri = (int)(item / P.ntile);
        const int t = (int)(item - (long long)ri * P.ntile);
        const int2 bs = P.rows[ri];
        const int b = bs.x, slot = bs.y;
        const ReqInfo rq = P.req[b];
        const char *row = row_ptr(P, b, slot, Fmt<DT>::kESZ);
        const long long ebase = (long long)t * TE;
        uint4 v[kVecPerThread];
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j)
            v[j] = load_vec<DT, VEC>(row, ebase + (long long)(j * kThreads + tid) * EPV, P.V);
        float tmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < kVecPerThread; ++j) tmax = fmaxf(tmax, vec_max<DT>(v[j]));
        float4 out;
        if (rq.greedy) {
            int idx = INT_MAX;
#pragma unroll
            for (int j = 0; j < kVecPerThread; ++j) {
#pragma unroll
                for (int i = 0; i < EPV; ++i) {
                    int e = (int)(ebase + (long long)(j * kThreads + tid) * EPV + i);
                    if (idx == INT_MAX && elem<DT>(v[j], i) == tmax) idx = e;
                }
            }
            float m = tmax;
            cta_argmax(m, idx, red_f, red_i);
            out = make_float4(m, 0.f, 0.f, __int_as_float(idx));
        } else {
            const float m = cta_max(tmax, red_f);
            FF s{0.f, 0.f};
            if (m > -INFINITY) {
                const float2 m2 = make_float2(m, m);
                const float2 chi = make_float2(rq.c_hi, rq.c_hi);
                const float2 clo = make_float2(rq.c_lo, rq.c_lo);
                BiasAcc2 acc;
                acc.init(1.0f);
#pragma unroll
                for (int j = 0; j < kVecPerThread; ++j) {
#pragma unroll
                    for (int i = 0; i < EPV; i += 2) {
                        float2 z = make_float2(elem<DT>(v[j], i), elem<DT>(v[j], i + 1));
                        acc.add(weight2(z, m2, chi, clo));
                    }
                }
                s = acc.total();
            }
            s = cta_sum_ff(s, red_f);
            out = make_float4(m, s.hi, s.lo, __int_as_float(-1));
        }
        if (tid == 0) P.stats[((size_t)b * P.nslot + slot) * P.ntile + t] = out;
    }
}

// ------------------------------------------------------------------ 3. decide

struct RowComb {
    float m;   // raw max logit of the row
    double S;  // sum_v 2^((z_v - m) c)
    int amax;  // lowest-index argmax (greedy rows)
};

__device__ RowComb combine_row(const Params &P, int b, int slot, double c, bool want_sum) {
    const float4 *st = P.stats + ((size_t)b * P.nslot + slot) * P.ntile;
    RowComb r;
    r.m = -INFINITY;
    r.amax = 0;
    bool first = true;
    for (int t = 0; t < P.ntile; ++t) {
        float4 s = st[t];
        if (first || s.x > r.m) {
            r.m = s.x;
            r.amax = __float_as_int(s.w);
            first = false;
        }
    }
    r.S = 0.0;
    if (want_sum && r.m > -INFINITY) {
        for (int t = 0; t < P.ntile; ++t) {
            float4 s = st[t];
            if (s.x > -INFINITY) {
                double f = exp2(((double)s.x - (double)r.m) * c);
                r.S += ((double)s.y + (double)s.z) * f;
            }
        }
    }
    return r;
}

constexpr int kDecideThreads = 64;

template <int DT>
__global__ void __launch_bounds__(kDecideThreads) sv_decide(Params P) {
    const int b = blockIdx.x, tid = threadIdx.x;
    const int K = P.K;
    const ReqInfo rq = P.req[b];
    const int L = rq.L;
    const bool greedy = rq.greedy != 0;
    __shared__ float s_m[SPEC_MAX_K + 1];
    __shared__ double s_S[SPEC_MAX_K + 1];
    __shared__ int s_amax[SPEC_MAX_K + 1];
    __shared__ float s_md[SPEC_MAX_K];
    __shared__ double s_Sd[SPEC_MAX_K];
    __shared__ int s_a;
    if (tid <= L) {
        RowComb r = combine_row(P, b, tid, rq.c, !greedy);
        s_m[tid] = r.m;
        s_S[tid] = r.S;
        s_amax[tid] = r.amax;
    }
    if (!greedy && tid < L) {
        RowComb r = combine_row(P, b, K + 1 + tid, rq.c, true);
        s_md[tid] = r.m;
        s_Sd[tid] = r.S;
    }
    __syncthreads();
    if (tid < 32) {
        bool acc = true;
        if (tid < L) {
            const int x = P.tokens[(size_t)b * K + tid];
            if (greedy) {
                acc = (x == s_amax[tid]);
            } else {
                const float g = load_logit(row_ptr(P, b, tid, Fmt<DT>::kESZ), DT, x);
                const float gd = load_logit(row_ptr(P, b, K + 1 + tid, Fmt<DT>::kESZ), DT, x);
                const double p = s_S[tid] > 0.0 ? exp2(((double)g - (double)s_m[tid]) * rq.c) / s_S[tid] : 0.0;
                const double q = s_Sd[tid] > 0.0 ? exp2(((double)gd - (double)s_md[tid]) * rq.c) / s_Sd[tid] : 0.0;
                const double u = uniform_accept(P.seed, (uint32_t)b, (uint32_t)tid);
                acc = u * q < p;
                if (P.dbg_probs) {
                    P.dbg_probs[((size_t)b * K + tid) * 2 + 0] = p;
                    P.dbg_probs[((size_t)b * K + tid) * 2 + 1] = q;
                }
            }
        }
        const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc);
        const int a = rej ? min(__ffs(rej) - 1, L) : L;
        if (tid == 0) s_a = a;
    }
    __syncthreads();
    const int a = s_a;
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    for (int k = tid; k <= K; k += kDecideThreads) {
        int v = -1;
        if (k < a) v = P.tokens[(size_t)b * K + k];
        else if (k == a && greedy) v = s_amax[a];
        out[k] = v;
    }
    if (tid == 0) P.accept_len[b] = a;
    if (!greedy) {
        const int mode = a < L ? 1 : 2;
        const int slot_t = a, slot_d = K + 1 + a;
        const float4 *st = P.stats + ((size_t)b * P.nslot + slot_t) * P.ntile;
        const float4 *sd = P.stats + ((size_t)b * P.nslot + slot_d) * P.ntile;
        for (int t = tid; t < P.ntile; t += kDecideThreads) {
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 s = st[t];
            if (s.x > -INFINITY && s_S[a] > 0.0) {
                double f = exp2(((double)s.x - (double)s_m[a]) * rq.c);
                if (mode == 1) f /= s_S[a];
                FF ff = ff_from_double(f);
                o.x = ff.hi;
                o.y = ff.lo;
            }
            if (mode == 1) {
                float4 d = sd[t];
                if (d.x > -INFINITY && s_Sd[a] > 0.0) {
                    double f = exp2(((double)d.x - (double)s_md[a]) * rq.c) / s_Sd[a];
                    FF ff = ff_from_double(f);
                    o.z = ff.hi;
                    o.w = ff.lo;
                }
            }
            P.alpha[(size_t)b * P.ntile + t] = o;
        }
        if (tid == 0) {
            SampInfo si;
            si.mode = mode;
            si.slot_t = slot_t;
            si.slot_d = slot_d;
            si.a = a;
            si.u = uniform_sample(P.seed, (uint32_t)b, (uint32_t)a);
            P.samp[b] = si;
        }
    } else if (tid == 0) {
        SampInfo si;
        si.mode = 0; si.slot_t = 0; si.slot_d = 0; si.a = a; si.u = 0.0;
        P.samp[b] = si;
    }
    if (P.dbg_rows) {
        const int nslot = 2 * K + 1;
        for (int s = tid; s < nslot; s += kDecideThreads) {
            double m = NAN, ls = NAN;
            if (!greedy) {
                if (s <= L) { m = (double)s_m[s] * rq.inv_t; ls = log(s_S[s]); }
                else if (s >= K + 1 && s - K - 1 < L) {
                    m = (double)s_md[s - K - 1] * rq.inv_t; ls = log(s_Sd[s - K - 1]);
                }
            }
            P.dbg_rows[((size_t)b * nslot + s) * 2 + 0] = m;
            P.dbg_rows[((size_t)b * nslot + s) * 2 + 1] = ls;
        }
        if (P.dbg_probs && greedy)
            for (int k = tid; k < K; k += kDecideThreads) {
                P.dbg_probs[((size_t)b * K + k) * 2 + 0] = NAN;
                P.dbg_probs[((size_t)b * K + k) * 2 + 1] = NAN;
            }
        if (P.dbg_probs && !greedy)
            for (int k = L + tid; k < K; k += kDecideThreads) {
                P.dbg_probs[((size_t)b * K + k) * 2 + 0] = NAN;
                P.dbg_probs[((size_t)b * K + k) * 2 + 1] = NAN;
            }
    }
}

// ------------------------------------------------------------------ 4/5. sampler

// Sampling weights of one 16-byte vector: w[i] = max(0, p - q) (residual) or
// p (bonus / fallback), with p = e * alpha_t and q = e' * alpha'_t formed from
// the same per-element weights as the statistics pass.
template <int DT>
__device__ __forceinline__ void vec_weights(const uint4 &vt, const uint4 &vd, bool resid,
                                            float2 m2, float2 md2, float2 chi, float2 clo,
                                            float2 ahi, float2 alo, float2 dhi, float2 dlo,
                                            float (&r)[Fmt<DT>::kEPV], float (&p)[Fmt<DT>::kEPV]) {
    constexpr int EPV = Fmt<DT>::kEPV;
#pragma unroll
    for (int i = 0; i < EPV; i += 2) {
        float2 e = weight2(make_float2(elem<DT>(vt, i), elem<DT>(vt, i + 1)), m2, chi, clo);
        float2 pp = fma2(e, ahi, mul2(e, alo));
        p[i] = pp.x;
        p[i + 1] = pp.y;
        if (resid) {
            float2 ed = weight2(make_float2(elem<DT>(vd, i), elem<DT>(vd, i + 1)), md2, chi, clo);
            float2 qq = fma2(ed, dhi, mul2(ed, dlo));
            float2 dd = sub2(pp, qq);
            r[i] = fmaxf(dd.x, 0.f);
            r[i + 1] = fmaxf(dd.y, 0.f);
        } else {
            r[i] = pp.x;
            r[i + 1] = pp.y;
        }
    }
}

template <int EPV>
__device__ __forceinline__ float seq_sum(const float (&w)[EPV]) {
    float s = w[0];
#pragma unroll
    for (int i = 1; i < EPV; ++i) s = __fadd_rn(s, w[i]);
    return s;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sv_sampletile(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int TE = tile_elems<DT>();
    __shared__ float red_f[2 * kWarps];
    const int tid = threadIdx.x;
    const long long total = (long long)P.B * P.ntile;
    for (long long item = blockIdx.x; item < total; item += gridDim.x) {
        const int b = (int)(item / P.ntile);
        const int t = (int)(item - (long long)b * P.ntile);
        const SampInfo si = P.samp[b];
        if (si.mode == 0) continue;
        const ReqInfo rq = P.req[b];
        const bool resid = si.mode == 1;
        const float mt = P.stats[((size_t)b * P.nslot + si.slot_t) * P.ntile + t].x;
        const float md = resid ? P.stats[((size_t)b * P.nslot + si.slot_d) * P.ntile + t].x : 0.f;
        const float4 al = P.alpha[(size_t)b * P.ntile + t];
        const char *rowt = row_ptr(P, b, si.slot_t, Fmt<DT>::kESZ);
        const char *rowd = resid ? row_ptr(P, b, si.slot_d, Fmt<DT>::kESZ) : rowt;
        const long long ebase = (long long)t * TE;
        const float2 m2 = make_float2(mt, mt), md2 = make_float2(md, md);
        const float2 chi = make_float2(rq.c_hi, rq.c_hi), clo = make_float2(rq.c_lo, rq.c_lo);
        const float2 ahi = make_float2(al.x, al.x), alo = make_float2(al.y, al.y);
        const float2 dhi = make_float2(al.z, al.z), dlo = make_float2(al.w, al.w);
        BiasAcc2 acc;  // .x residual, .y p
        acc.init(16.0f);
#pragma unroll 2
        for (int j = 0; j < kVecPerThread; ++j) {
            const long long e0 = ebase + (long long)(j * kThreads + tid) * EPV;
            const uint4 vt = load_vec<DT, VEC>(rowt, e0, P.V);
            const uint4 vd = resid ? load_vec<DT, VEC>(rowd, e0, P.V) : vt;
            float r[EPV], p[EPV];
            vec_weights<DT>(vt, vd, resid, m2, md2, chi, clo, ahi, alo, dhi, dlo, r, p);
            acc.add(make_float2(seq_sum<EPV>(r), seq_sum<EPV>(p)));
        }
        FF zr{__fsub_rn(acc.h.x, 16.0f), acc.l.x};
        FF zp{__fsub_rn(acc.h.y, 16.0f), acc.l.y};
        zr = cta_sum_ff(ff_add(zr, FF{0.f, 0.f}), red_f);
        zp = cta_sum_ff(ff_add(zp, FF{0.f, 0.f}), red_f);
        if (tid == 0) P.ztile[(size_t)b * P.ntile + t] = make_float4(zr.hi, zr.lo, zp.hi, zp.lo);
    }
}

// CTA-wide exclusive prefix sum of doubles; `tot` receives the total.
__device__ __forceinline__ double cta_excl_scan(double v, double *red, double &tot) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    double excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) excl = 0.0;
    __syncthreads();
    if (lane == 31) red[w] = incl;
    __syncthreads();
    double off = 0.0;
    for (int i = 0; i < w; ++i) off += red[i];
    tot = 0.0;
    for (int i = 0; i < kWarps; ++i) tot += red[i];
    return off + excl;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) sv_find(Params P) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int TE = tile_elems<DT>();
    __shared__ double red_d[kWarps];
    __shared__ int s_tok;
    __shared__ float red_f[2 * kWarps];
    __shared__ int red_i[kWarps];
    const int b = blockIdx.x, tid = threadIdx.x;
    const SampInfo si = P.samp[b];
    if (si.mode == 0) return;
    const ReqInfo rq = P.req[b];
    // tile masses
    double Zr = 0.0, Zp = 0.0;
    for (int t = 0; t < P.ntile; ++t) {
        float4 z = P.ztile[(size_t)b * P.ntile + t];
        Zr += (double)z.x + (double)z.y;
        Zp += (double)z.z + (double)z.w;
    }
    const bool use_r = si.mode == 1 && Zr > 0.0;
    const double Z = use_r ? Zr : Zp;
    const double theta = si.u * Z;
    int tsel = -1, tlast = P.ntile - 1;
    double cum = 0.0;
    for (int t = 0; t < P.ntile; ++t) {
        float4 z = P.ztile[(size_t)b * P.ntile + t];
        double zt = use_r ? (double)z.x + (double)z.y : (double)z.z + (double)z.w;
        if (zt > 0.0) tlast = t;
        if (tsel < 0 && cum + zt > theta) tsel = t;
        if (tsel < 0) cum += zt;
    }
    double th_local = INFINITY;
    if (tsel >= 0) th_local = theta - cum;
    else tsel = tlast;
    const int t = tsel;
    const bool resid = si.mode == 1;
    const float mt = P.stats[((size_t)b * P.nslot + si.slot_t) * P.ntile + t].x;
    const float md = resid ? P.stats[((size_t)b * P.nslot + si.slot_d) * P.ntile + t].x : 0.f;
    const float4 al = P.alpha[(size_t)b * P.ntile + t];
    const char *rowt = row_ptr(P, b, si.slot_t, Fmt<DT>::kESZ);
    const char *rowd = resid ? row_ptr(P, b, si.slot_d, Fmt<DT>::kESZ) : rowt;
    const long long ebase = (long long)t * TE;
    const float2 m2 = make_float2(mt, mt), md2 = make_float2(md, md);
    const float2 chi = make_float2(rq.c_hi, rq.c_hi), clo = make_float2(rq.c_lo, rq.c_lo);
    const float2 ahi = make_float2(al.x, al.x), alo = make_float2(al.y, al.y);
    const float2 dhi = make_float2(al.z, al.z), dlo = make_float2(al.w, al.w);
    if (tid == 0) s_tok = INT_MAX;
    double base = 0.0;
    int last_pos = -1;  // largest index with positive weight seen by this thread
    for (int j = 0; j < kVecPerThread; ++j) {
        const long long e0 = ebase + (long long)(j * kThreads + tid) * EPV;
        const uint4 vt = load_vec<DT, VEC>(rowt, e0, P.V);
        const uint4 vd = resid ? load_vec<DT, VEC>(rowd, e0, P.V) : vt;
        float r[EPV], p[EPV], w[EPV];
        vec_weights<DT>(vt, vd, resid, m2, md2, chi, clo, ahi, alo, dhi, dlo, r, p);
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
            w[i] = use_r ? r[i] : p[i];
            if (w[i] > 0.f && e0 + i < P.V) last_pos = (int)(e0 + i);
        }
        const float sv = seq_sum<EPV>(w);
        double tot;
        const double col = base + cta_excl_scan((double)sv, red_d, tot);
        if (col <= th_local && col + (double)sv > th_local) {
            float ps = 0.f;
            int tok = -1;
#pragma unroll
            for (int i = 0; i < EPV; ++i) {
                ps = i == 0 ? w[0] : __fadd_rn(ps, w[i]);
                if (tok < 0 && col + (double)ps > th_local) tok = (int)(e0 + i);
            }
            if (tok >= 0) atomicMin(&s_tok, tok);
        }
        base += tot;
        __syncthreads();
        if (s_tok != INT_MAX) break;
    }
    int tok = s_tok;
    if (tok == INT_MAX) {
        // rounding left no crossing: largest index with positive weight
        float v = last_pos >= 0 ? 1.f : 0.f;
        int idx = last_pos >= 0 ? -last_pos : INT_MAX;
        cta_argmax(v, idx, red_f, red_i);
        tok = (v > 0.f) ? -idx : (int)ebase;
    }
    if (tid == 0) P.out_tokens[(size_t)b * (P.K + 1) + si.a] = tok;
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
    size_t req, row_count, rows, stats, samp, alpha, ztile, total;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int tile_elems_for(spec_dtype_t dt) {
    return dt == SPEC_DTYPE_BF16 ? tile_elems<kBF16>() : tile_elems<kF32>();
}

static bool sizes_ok(int B, int K, int V) {
    return B >= 1 && B < (1 << 24) && K >= 1 && K <= SPEC_MAX_K && V >= 2 && V <= SPEC_MAX_V;
}

static Layout layout(int B, int K, int V, spec_dtype_t dt) {
    Layout L{};
    const size_t ntile = (size_t)((V + tile_elems_for(dt) - 1) / tile_elems_for(dt));
    const size_t nslot = (size_t)(2 * K + 1);
    size_t off = 0;
    L.req = off; off = align256(off + sizeof(ReqInfo) * (size_t)B);
    L.row_count = off; off = align256(off + sizeof(int));
    L.rows = off; off = align256(off + sizeof(int2) * (size_t)B * nslot);
    L.stats = off; off = align256(off + sizeof(float4) * (size_t)B * nslot * ntile);
    L.samp = off; off = align256(off + sizeof(SampInfo) * (size_t)B);
    L.alpha = off; off = align256(off + sizeof(float4) * (size_t)B * ntile);
    L.ztile = off; off = align256(off + sizeof(float4) * (size_t)B * ntile);
    L.total = off;
    return L;
}

struct DevInfo {
    int sms = 0;
    int occ_stats[2][2] = {{0, 0}, {0, 0}};
    int occ_tile[2][2] = {{0, 0}, {0, 0}};
};

static DevInfo g_dev[64];

template <int DT, bool VEC>
static void occ_for(DevInfo &d) {
    int o = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_rowstats<DT, VEC>, kThreads, 0);
    d.occ_stats[DT][VEC] = o > 0 ? o : 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sv_sampletile<DT, VEC>, kThreads, 0);
    d.occ_tile[DT][VEC] = o > 0 ? o : 1;
}

static const DevInfo *dev_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    DevInfo &d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        occ_for<kF32, false>(d);
        occ_for<kF32, true>(d);
        occ_for<kBF16, false>(d);
        occ_for<kBF16, true>(d);
        d.sms = sms;
    }
    return &d;
}

static cudaEvent_t g_prof_start = nullptr, g_prof_end = nullptr;
constexpr int kKernelsPerVerify = 5;

template <int DT, bool VEC>
static void launch_all(const Params &P, const DevInfo &d, cudaStream_t s) {
    sv_prep<<<1, kPrepThreads, 0, s>>>(P);
    const int g1 = d.sms * d.occ_stats[DT][VEC];
    if (g_prof_start) cudaEventRecord(g_prof_start, s);
    sv_rowstats<DT, VEC><<<g1, kThreads, 0, s>>>(P);
    if (g_prof_end) cudaEventRecord(g_prof_end, s);
    sv_decide<DT><<<P.B, kDecideThreads, 0, s>>>(P);
    const long long items = (long long)P.B * P.ntile;
    long long g2 = (long long)d.sms * d.occ_tile[DT][VEC];
    if (g2 > items) g2 = items;
    sv_sampletile<DT, VEC><<<(int)g2, kThreads, 0, s>>>(P);
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
    P.ntile = (V + tile_elems_for(dtype) - 1) / tile_elems_for(dtype);
    P.nslot = 2 * K + 1;
    P.out_tokens = out_tokens;
    P.accept_len = accept_len;
    P.dev_status = dev_status;
    P.dbg_rows = row_stats;
    P.dbg_probs = probs;
    char *ws = static_cast<char *>(workspace);
    P.req = reinterpret_cast<ReqInfo *>(ws + L.req);
    P.row_count = reinterpret_cast<int *>(ws + L.row_count);
    P.rows = reinterpret_cast<int2 *>(ws + L.rows);
    P.stats = reinterpret_cast<float4 *>(ws + L.stats);
    P.samp = reinterpret_cast<SampInfo *>(ws + L.samp);
    P.alpha = reinterpret_cast<float4 *>(ws + L.alpha);
    P.ztile = reinterpret_cast<float4 *>(ws + L.ztile);
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
