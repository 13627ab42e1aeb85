// sv_fused.cuh -- the fused, persistent verification kernel (16-byte aligned rows).
//
// One launch streams every needed logit row once and finishes every request
// inside the same grid, so the row (pair) a rejected request samples from is
// re-read while it is still resident in L2:
//
//   producer warps (two per CTA)     consumer warps (kFC per CTA)
//   ------------------------------   ---------------------------------------------
//   warp 0: claims stream items in   claim the next stage, wait for its bytes,
//   batches of 32 from a global      copy it to registers, release it, then:
//   counter, gathers their row         stream item  -> chunk partial; the last
//   metadata across its lanes and      chunk of a row combines the row; the last
//   bulk-copies each 8 KiB item        row of a request decides it (acceptance
//   into the next free stage           rule, first rejection, outputs) and
//   warp 1: claims sampler tasks in    publishes its sampler tasks
//   batches (atomic add), waits for    sampler task -> residual / target masses
//   their request, copies each 4 KiB   of a 4 KiB chunk of the row (pair); the
//   chunk of the row (pair)            last task of a request draws the token
//   both allocate stages from one      (inverse CDF)
//   shared sequence counter
//
// Work order is request-major, so the rows of a request are read within a short
// window and a request's sampler tasks find its rows in L2.  Every wait is
// bounded (SPEC_DEV_TIMEOUT is raised on expiry).  Work is claimed from global
// counters, never owned in advance, so CTAs that are not resident yet hold no
// work that resident ones wait for.
#pragma once
#include "sv_common.cuh"

namespace sv {

constexpr int kFC = 4;                         // consumer warps per CTA
constexpr int kFProd = 2;                      // producer warps per CTA
constexpr int kFThreads = (kFC + kFProd) * 32;
constexpr int kFStages = 2 * kFC;              // shared-memory stages per CTA
// Stage sequence number k goes to stage k % kFStages and to consumer warp
// k % kFC, so every stage is consumed in order by one warp and filled in order
// under the producers' lock: no barrier is ever more than one phase away from
// the phase its waiter names (1-bit parity waits stay unambiguous).
static_assert(kFStages % kFC == 0, "stages must be a multiple of the consumers");
constexpr int kStageBytes = 8192;              // one stream item / one sampler task
constexpr int kStreamVec = kStageBytes / 16 / 32;  // 16 vectors per lane
constexpr int kSubBytes = 4096;                // per row of a sampler task
constexpr int kSubVec = kSubBytes / 16 / 32;   // 8 vectors per lane

enum { kKindStream = 0, kKindSample = 1, kKindEnd = 2 };

struct Desc {
    int kind, b, slot, c;
    int nvec;     // valid 16-byte vectors of the (first) row
    float cval;   // log2(e)/T as float (stream items)
    int greedy;
    int pad;
};

struct FusedShared {
    uint4 buf[kFStages][kStageBytes / 16];
    Desc desc[kFStages];
    unsigned long long full[kFStages];
    unsigned long long empty[kFStages];
    unsigned int prod_seq;  // producer stage sequence (under prod_lock)
    unsigned int prod_done; // producers finished
    int prod_lock;          // serialises stage allocation + fill between producers
};

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ int ld_volatile_int(const int *p) {
    return *reinterpret_cast<const volatile int *>(p);
}

// acc += (2^((lo(w) - m) c), 2^((hi(w) - m) c)) for the two bfloat16 of w.
__device__ __forceinline__ void bf16x2_exp_acc(uint32_t w, unsigned long long m2,
                                               unsigned long long c2, unsigned long long &acc) {
    asm("{\n\t.reg .b32 a, b;\n\t.reg .b64 z;\n\t"
        "shl.b32 a, %1, 16;\n\tand.b32 b, %1, 0xFFFF0000;\n\tmov.b64 z, {a, b};\n\t"
        "sub.rn.f32x2 z, z, %2;\n\tmul.rn.f32x2 z, z, %3;\n\t"
        "mov.b64 {a, b}, z;\n\tex2.approx.ftz.f32 a, a;\n\tex2.approx.ftz.f32 b, b;\n\t"
        "mov.b64 z, {a, b};\n\tadd.rn.f32x2 %0, %0, z;\n\t}"
        : "+l"(acc)
        : "r"(w), "l"(m2), "l"(c2));
}

// Same for two float32 logits.
__device__ __forceinline__ void f32x2_exp_acc(uint32_t w0, uint32_t w1, unsigned long long m2,
                                              unsigned long long c2, unsigned long long &acc) {
    asm("{\n\t.reg .b32 a, b;\n\t.reg .b64 z;\n\t"
        "mov.b64 z, {%1, %2};\n\t"
        "sub.rn.f32x2 z, z, %3;\n\tmul.rn.f32x2 z, z, %4;\n\t"
        "mov.b64 {a, b}, z;\n\tex2.approx.ftz.f32 a, a;\n\tex2.approx.ftz.f32 b, b;\n\t"
        "mov.b64 z, {a, b};\n\tadd.rn.f32x2 %0, %0, z;\n\t}"
        : "+l"(acc)
        : "r"(w0), "r"(w1), "l"(m2), "l"(c2));
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// SampInfo written by another SM during this kernel: read it from L2.
__device__ __forceinline__ SampInfo load_samp(const Params &P, int b) {
    static_assert(sizeof(SampInfo) % 16 == 0, "SampInfo layout");
    SampInfo si;
    const int4 *src = reinterpret_cast<const int4 *>(P.samp + b);
    int4 *dst = reinterpret_cast<int4 *>(&si);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(SampInfo) / 16); ++i) dst[i] = __ldcg(src + i);
    return si;
}

// ------------------------------------------------------------------ stream item

// Chunk partial of one stream item held in registers (lane's vector i is
// vector i*32 + lane of the chunk): greedy rows {max, -, -, lowest argmax},
// sampled rows {max, sum 2^((z - max) c), -, -1}.
template <int DT>
__device__ __forceinline__ float4 stream_partial(const uint4 (&v)[kStreamVec], int nvec, bool greedy,
                                                 float c, int e0, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    float lm = -INFINITY;
    if (DT == kBF16) {
        uint32_t run = 0xFF80FF80u;
#pragma unroll
        for (int i = 0; i < kStreamVec; ++i) {
            if (i * 32 + lane < nvec) {
                run = bf16x2_max(run, bf16x2_max(bf16x2_max(v[i].x, v[i].y), bf16x2_max(v[i].z, v[i].w)));
            }
        }
        lm = fmaxf(__uint_as_float(run << 16), __uint_as_float(run & 0xFFFF0000u));
    } else {
#pragma unroll
        for (int i = 0; i < kStreamVec; ++i)
            if (i * 32 + lane < nvec) lm = fmaxf(lm, vec_max<DT>(v[i]));
    }
    const float m = warp_max(lm);
    if (greedy) {
        int idx = INT_MAX;
        if (lm == m) {
#pragma unroll
            for (int i = 0; i < kStreamVec; ++i) {
                if (i * 32 + lane < nvec) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (idx == INT_MAX && elem<DT>(v[i], e) == m) idx = e0 + (i * 32 + lane) * EPV + e;
                }
            }
        }
        return make_float4(m, 0.f, 0.f, __int_as_float(warp_min_int(idx)));
    }
    float s = 0.f;
    if (m > -INFINITY) {
        const unsigned long long m2 = f2u(make_float2(m, m)), c2 = f2u(make_float2(c, c));
        unsigned long long a0 = 0ull, a1 = 0ull;
#pragma unroll
        for (int i = 0; i < kStreamVec; ++i) {
            if (i * 32 + lane < nvec) {
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
        s = t.x + t.y;
    }
    return make_float4(m, warp_sum(s), 0.f, __int_as_float(-1));
}

// ------------------------------------------------------------------ row combine

// Row statistics from its chunk partials (one warp): {max, S (sampled) or 0,
// lowest argmax (greedy) as int bits, -}.
__device__ __forceinline__ float4 combine_row(const Params &P, int b, int slot, bool greedy,
                                              float c, int lane) {
    const float4 *pp = P.part + ((size_t)b * P.nslot + slot) * P.nchunk8;
    float m = -INFINITY;
    for (int i = lane; i < P.nchunk8; i += 32) m = fmaxf(m, __ldcg(&pp[i].x));
    m = warp_max(m);
    if (greedy) {
        int amax = INT_MAX;
        for (int i = lane; i < P.nchunk8; i += 32) {
            const float4 q = __ldcg(&pp[i]);
            if (q.x == m) amax = min(amax, __float_as_int(q.w));
        }
        return make_float4(m, 0.f, __int_as_float(warp_min_int(amax)), 0.f);
    }
    float S = 0.f;
    if (m > -INFINITY)
        for (int i = lane; i < P.nchunk8; i += 32) {
            const float4 q = __ldcg(&pp[i]);
            if (q.x > -INFINITY) S += q.y * ex2((q.x - m) * c);
        }
    return make_float4(m, warp_sum(S), __int_as_float(-1), 0.f);
}

// ------------------------------------------------------------------ decide

// Acceptance decision of request b by one warp (lane k = draft position k).
template <int DT>
__device__ __noinline__ void decide_request(const Params &P, int b, int lane) {
    const int K = P.K;
    const ReqInfo rq = P.req[b];
    const int L = rq.L;
    const bool greedy = rq.greedy != 0;
    const float4 *rs = P.rowstat + (size_t)b * P.nslot;
    float4 rt = make_float4(0.f, 0.f, 0.f, 0.f), rd = rt;
    if (lane <= L) rt = __ldcg(&rs[lane]);
    if (!greedy && lane < L) rd = __ldcg(&rs[K + 1 + lane]);
    bool acc = true;
    double p = NAN, q = NAN;
    if (lane < L) {
        const int x = P.tokens[(size_t)b * K + lane];
        if (greedy) {
            acc = (x == __float_as_int(rt.z));
        } else {
            const float g = load_logit(row_ptr(P, b, lane, Fmt<DT>::kESZ), DT, x);
            const float gd = load_logit(row_ptr(P, b, K + 1 + lane, Fmt<DT>::kESZ), DT, x);
            p = rt.y > 0.f ? exp2(((double)g - (double)rt.x) * rq.cd) / (double)rt.y : 0.0;
            q = rd.y > 0.f ? exp2(((double)gd - (double)rd.x) * rq.cd) / (double)rd.y : 0.0;
            const double u = uniform_accept(P.seed, (uint32_t)b, (uint32_t)lane);
            acc = u * q < p;
        }
    }
    const unsigned rej = ~__ballot_sync(0xFFFFFFFFu, acc);
    const int a = rej ? min(__ffs(rej) - 1, L) : L;
    // row statistics of row a (held by lane a; a <= L <= K <= 32: lane 32 is K=32,L=32)
    const float4 ra = a < 32 ? make_float4(__shfl_sync(0xFFFFFFFFu, rt.x, a & 31),
                                           __shfl_sync(0xFFFFFFFFu, rt.y, a & 31),
                                           __shfl_sync(0xFFFFFFFFu, rt.z, a & 31), 0.f)
                             : __ldcg(&rs[a]);
    const float4 rda = (a < 32) ? make_float4(__shfl_sync(0xFFFFFFFFu, rd.x, a & 31),
                                              __shfl_sync(0xFFFFFFFFu, rd.y, a & 31), 0.f, 0.f)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    for (int k = lane; k <= K; k += 32) {
        int v = -1;
        if (k < a) v = P.tokens[(size_t)b * K + k];
        else if (k == a && greedy) v = __float_as_int(ra.z);
        out[k] = v;
    }
    if (P.dbg_probs && lane < K) {  // lane k holds position k (K <= 32)
        P.dbg_probs[((size_t)b * K + lane) * 2 + 0] = (!greedy && lane < L) ? p : NAN;
        P.dbg_probs[((size_t)b * K + lane) * 2 + 1] = (!greedy && lane < L) ? q : NAN;
    }
    if (P.dbg_rows) {
        const int nslot = 2 * K + 1;
        for (int sl = lane; sl < nslot; sl += 32) {
            double m = NAN, ls = NAN;
            if (!greedy && (sl <= L || (sl >= K + 1 && sl - K - 1 < L))) {
                const float4 r = __ldcg(&rs[sl]);
                m = (double)r.x * rq.inv_t;
                ls = log((double)r.y);
            }
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 0] = m;
            P.dbg_rows[((size_t)b * nslot + sl) * 2 + 1] = ls;
        }
    }
    if (lane == 0) {
        P.accept_len[b] = a;
        if (!greedy) {
            SampInfo si;
            si.mode = a < L ? 1 : 2;
            si.a = a;
            si.slot_t = a;
            si.slot_d = K + 1 + a;
            si.m_t = ra.x;
            si.rho_t = 1.f;
            si.m_d = 0.f;
            si.rho_d = 0.f;
            if (si.mode == 1) {
                si.rho_t = 1.f / ra.y;
                si.m_d = rda.x;
                si.rho_d = 1.f / rda.y;
            }
            si.c_hi = rq.c_hi;
            si.c_lo = rq.c_lo;
            si.pad0 = si.pad1 = 0;
            si.u = uniform_sample(P.seed, (uint32_t)b, (uint32_t)a);
            si.pad2 = 0.0;
            P.samp[b] = si;
            __threadfence();
            const int e = atomicAdd(P.q_alloc, 1);
            *reinterpret_cast<volatile int *>(&P.q_entries[e]) = b + 1;
            __threadfence();
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------------ sampler task

// Masses of one 4 KiB chunk of the sampled row (pair), see sv_sample.
template <int DT>
__device__ __forceinline__ void sample_masses(const uint4 (&vt)[kSubVec], const uint4 (&vd)[kSubVec],
                                              int nvec, const SampInfo &si, float &A, float &Bs,
                                              float &W, FF &st, FF &sd, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    const float2 m2 = make_float2(si.m_t, si.m_d);
    const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
    const float2 rho2 = make_float2(si.rho_t, si.rho_d);
    BiasAcc2 acc;
    acc.init(1.0f);
    A = 0.f; Bs = 0.f; W = 0.f;
#pragma unroll
    for (int i = 0; i < kSubVec; ++i) {
        if (i * 32 + lane < nvec) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                const float2 ee = weight2(make_float2(elem<DT>(vt[i], e), elem<DT>(vd[i], e)), m2, chi2, clo2);
                const float2 ab = mul2(ee, rho2);
                acc.add(ee);
                W = __fadd_rn(W, ab.x);
                if (ab.x > ab.y) {
                    A = __fadd_rn(A, ab.x);
                    Bs = __fadd_rn(Bs, ab.y);
                }
            }
        }
    }
    A = warp_sum(A);
    Bs = warp_sum(Bs);
    W = warp_sum(W);
    st = warp_sum_ff(ff_add(FF{__fsub_rn(acc.h.x, 1.0f), acc.l.x}, FF{0.f, 0.f}));
    sd = warp_sum_ff(ff_add(FF{__fsub_rn(acc.h.y, 1.0f), acc.l.y}, FF{0.f, 0.f}));
}

// ------------------------------------------------------------------ inverse CDF (one warp)

template <int DT>
__device__ __noinline__ void find_request(const Params &P, int b, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = kSubBytes / ESZ;
    const SampInfo si = load_samp(P, b);
    const bool resid = si.mode == 1;
    const int nch = P.nsub;
    const float4 *sub = P.sub + (size_t)b * nch;
    const float4 *sex = P.sexact + (size_t)b * nch;
    double st = 0.0, sd = 0.0, zw = 0.0;
    for (int c = lane; c < nch; c += 32) {
        const float4 e = __ldcg(&sex[c]);
        st += (double)e.x + (double)e.y;
        sd += (double)e.z + (double)e.w;
    }
    st = warp_sum_d(st);
    sd = warp_sum_d(sd);
    const double kt = resid ? 1.0 / ((double)si.rho_t * st) : 1.0;
    const double kd = resid ? 1.0 / ((double)si.rho_d * sd) : 0.0;
    // contiguous block of chunks per lane
    const int per = (nch + 31) / 32;
    const int c0 = lane * per, c1 = min(nch, c0 + per);
    double zr = 0.0;
    for (int c = c0; c < c1; ++c) {
        const float4 q = __ldcg(&sub[c]);
        zr += resid ? fmax(0.0, kt * (double)q.x - kd * (double)q.y) : (double)q.z;
        zw += (double)q.z;
    }
    const double Zr = warp_sum_d(zr), Zw = warp_sum_d(zw);
    const bool use_w = !resid || !(Zr > 0.0);
    const double Z = use_w ? Zw : Zr;
    const double theta = si.u * Z;
    const double mine = use_w ? zw : zr;
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    double base = incl - mine;
    int my_c = INT_MAX;
    double my_base = 0.0;
    if (base <= theta && base + mine > theta) {
        for (int c = c0; c < c1; ++c) {
            const float4 q = __ldcg(&sub[c]);
            const double v = use_w ? (double)q.z : fmax(0.0, kt * (double)q.x - kd * (double)q.y);
            if (base + v > theta) {
                my_c = c;
                my_base = base;
                break;
            }
            base += v;
        }
    }
    const int ch_found = warp_min_int(my_c);
    int ch;
    double th_local;
    if (ch_found != INT_MAX) {
        ch = ch_found;
        const int owner = __ffs(__ballot_sync(0xFFFFFFFFu, my_c == ch_found)) - 1;
        th_local = theta - __shfl_sync(0xFFFFFFFFu, my_base, owner);
    } else {
        // rounding left no crossing: the last chunk with positive mass
        int last = -1;
        for (int c = c0; c < c1; ++c) {
            const float4 q = __ldcg(&sub[c]);
            const double v = use_w ? (double)q.z : fmax(0.0, kt * (double)q.x - kd * (double)q.y);
            if (v > 0.0) last = c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xFFFFFFFFu, last, o));
        ch = last >= 0 ? last : nch - 1;
        th_local = INFINITY;
    }
    const char *rowt = row_ptr(P, b, si.slot_t, ESZ);
    const char *rowd = resid ? row_ptr(P, b, si.slot_d, ESZ) : rowt;
    const long long e0 = (long long)ch * CE;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const float2 m2 = make_float2(si.m_t, si.m_d);
    const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
    const float2 rho2 = (resid && !use_w) ? make_float2(si.rho_t, si.rho_d) : make_float2(si.rho_t, 0.f);
    const float dkt = (float)(kt - 1.0), dkd = (float)(kd - 1.0);
    double run = 0.0;
    int found = INT_MAX, last_pos = -1;
    for (int i = 0; i < kSubVec && found == INT_MAX; ++i) {
        const long long q0 = e0 + (long long)(i * 32 + lane) * EPV;
        const uint4 vt = load_vec<DT, true>(rowt, q0, P.V);
        const uint4 vd = (resid && !use_w) ? load_vec<DT, true>(rowd, q0, P.V) : make_uint4(ni, ni, ni, ni);
        float w[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
            const float2 ee = weight2(make_float2(elem<DT>(vt, e), elem<DT>(vd, e)), m2, chi2, clo2);
            const float2 ab = mul2(ee, rho2);
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

// ------------------------------------------------------------------ producer helpers

// Producer lock: stage allocation, the wait for the stage's release and the
// fill happen in sequence order.  Bounded; returns false on timeout.
__device__ __forceinline__ bool prod_lock(FusedShared &sh) {
    if (atomicCAS(&sh.prod_lock, 0, 1) == 0) {
        __threadfence_block();
        return true;
    }
    const unsigned long long t0 = global_ns();
    for (;;) {
        __nanosleep(64);
        if (atomicCAS(&sh.prod_lock, 0, 1) == 0) {
            __threadfence_block();
            return true;
        }
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ void prod_unlock(FusedShared &sh) {
    __threadfence_block();
    atomicExch(&sh.prod_lock, 0);
}

// Next stage for a producer (caller holds the lock): allocate a sequence number
// and wait until the stage's previous contents have been released.
__device__ __forceinline__ bool acquire_stage(FusedShared &sh, uint32_t &k) {
    volatile unsigned int *seq = &sh.prod_seq;
    k = *seq;
    *seq = k + 1u;
    if (k < (uint32_t)kFStages) return true;
    return mbar_wait_bounded(reinterpret_cast<uint64_t *>(&sh.empty[k % kFStages]),
                             ((k / kFStages) - 1u) & 1u, kWaitLimitNs);
}

// The last producer to finish writes one end marker per consumer warp (kFC
// consecutive sequence numbers: one per consumer).
__device__ __forceinline__ void producer_done(const Params &P, FusedShared &sh) {
    if (atomicAdd(&sh.prod_done, 1u) != (unsigned)(kFProd - 1)) return;
    if (!prod_lock(sh)) {
        if (P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        return;
    }
    for (int j = 0; j < kFC; ++j) {
        uint32_t k;
        if (!acquire_stage(sh, k) && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        const int s = (int)(k % kFStages);
        Desc d;
        d.kind = kKindEnd; d.b = d.slot = d.c = d.nvec = d.greedy = d.pad = 0; d.cval = 0.f;
        sh.desc[s] = d;
        mbar_arrive(&sh.full[s]);
    }
    prod_unlock(sh);
}

constexpr int kStreamBatch = 32;  // stream items claimed per global atomic (one per lane)
constexpr int kTaskBatch = 16;    // sampler tasks claimed per global atomic (one per lane)
constexpr int kIssueGroup = 8;    // stages acquired per lock hold (<= kFStages)
static_assert(kIssueGroup <= kFStages, "issue group larger than the ring");

// Lane 0 takes the lock, allocates `nn` consecutive sequence numbers and waits,
// in order, until each of their stages has been released; the lock is then
// held until the group is issued (`group_end`).  Returns the first sequence
// number, or ~0u on timeout (lock released).
__device__ __forceinline__ uint32_t group_begin(FusedShared &sh, int nn, int lane) {
    uint32_t k0 = 0;
    int ok = 1;
    if (lane == 0) {
        ok = prod_lock(sh);
        if (ok) {
            volatile unsigned int *seq = &sh.prod_seq;
            k0 = *seq;
            *seq = k0 + (uint32_t)nn;
            for (int i = 0; i < nn && ok; ++i) {
                const uint32_t k = k0 + (uint32_t)i;
                if (k >= (uint32_t)kFStages &&
                    !mbar_wait_bounded(reinterpret_cast<uint64_t *>(&sh.empty[k % kFStages]),
                                       ((k / kFStages) - 1u) & 1u, kWaitLimitNs))
                    ok = 0;
            }
            if (!ok) prod_unlock(sh);
        }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    k0 = __shfl_sync(0xFFFFFFFFu, k0, 0);
    return ok ? k0 : ~0u;
}

__device__ __forceinline__ void group_end(FusedShared &sh, int lane) {
    __syncwarp();
    if (lane == 0) prod_unlock(sh);
}

template <int DT>
__device__ __noinline__ void stream_producer(const Params &P, FusedShared &sh, int lane) {
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE8 = kStageBytes / ESZ;
    const uint32_t n_stream = (uint32_t)(*P.row_count) * (uint32_t)P.nchunk8;
    for (;;) {
        uint32_t base = 0;
        if (lane == 0) base = atomicAdd(P.stream_head, (unsigned)kStreamBatch);
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        if (base >= n_stream) break;
        // metadata of the batch, one item per lane
        const uint32_t item = base + (uint32_t)lane;
        Desc d;
        d.kind = kKindStream; d.b = 0; d.slot = 0; d.c = 0; d.nvec = 0; d.cval = 0.f;
        d.greedy = 0; d.pad = 0;
        const char *src = nullptr;
        uint32_t bytes = 0;
        if (item < n_stream) {
            const uint32_t ri = item / (uint32_t)P.nchunk8;
            const uint32_t c = item - ri * (uint32_t)P.nchunk8;
            const int2 bs = P.rows[ri];
            const ReqInfo rq = P.req[bs.x];
            bytes = min((uint32_t)CE8, (uint32_t)P.V - c * CE8) * ESZ;
            d.b = bs.x; d.slot = bs.y; d.c = (int)c; d.nvec = (int)(bytes / 16);
            d.cval = rq.c; d.greedy = rq.greedy;
            src = row_ptr(P, bs.x, bs.y, ESZ) + (size_t)c * CE8 * ESZ;
        }
        const int n = (int)min((uint32_t)kStreamBatch, n_stream - base);
        for (int j0 = 0; j0 < n; j0 += kIssueGroup) {
            const int nn = min(kIssueGroup, n - j0);
            const uint32_t k0 = group_begin(sh, nn, lane);
            if (k0 == ~0u) {
                if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
                if (lane == 0) producer_done(P, sh);
                return;
            }
            if (lane >= j0 && lane < j0 + nn) {
                const int s = (int)((k0 + (uint32_t)(lane - j0)) % kFStages);
                sh.desc[s] = d;
                uint64_t *fb = reinterpret_cast<uint64_t *>(&sh.full[s]);
                mbar_expect_tx(fb, bytes);
                bulk_g2s(sh.buf[s], src, bytes, fb);
            }
            group_end(sh, lane);
        }
    }
    if (lane == 0) producer_done(P, sh);
}

// Sampler tasks: request entry e (publication order) owns task indices
// [e * nsub_pad, (e + 1) * nsub_pad), nsub_pad = nsub rounded up to kTaskBatch,
// so a claimed batch never straddles two requests.  Batches are claimed with
// one atomic add (no retries); a batch whose request is not published yet is
// waited for (bounded), which never blocks stream items: they have their own
// producer warp.  Lane i issues task c0 + i.
__device__ __noinline__ void task_producer(const Params &P, FusedShared &sh, int esz, int lane) {
    const int ce4 = kSubBytes / esz;
    const unsigned long long nsub_pad =
        (unsigned long long)((P.nsub + kTaskBatch - 1) / kTaskBatch) * kTaskBatch;
    const unsigned long long total = (unsigned long long)(*P.n_sampled) * nsub_pad;
    for (;;) {
        unsigned long long h = 0;
        if (lane == 0) h = atomicAdd(P.q_head, (unsigned long long)kTaskBatch);
        h = __shfl_sync(0xFFFFFFFFu, h, 0);
        if (h >= total) break;
        const unsigned long long e = h / nsub_pad;
        const int c0 = (int)(h - e * nsub_pad);
        int bp1 = 0;
        if (lane == 0) {
            bp1 = ld_volatile_int(&P.q_entries[e]);
            if (bp1 == 0) {
                const unsigned long long t0 = global_ns();
                unsigned int nap = 128;
                while ((bp1 = ld_volatile_int(&P.q_entries[e])) == 0) {
                    if (global_ns() - t0 > kWaitLimitNs) break;
                    __nanosleep(nap);
                    if (nap < 2048) nap <<= 1;
                }
            }
            __threadfence();
        }
        bp1 = __shfl_sync(0xFFFFFFFFu, bp1, 0);
        if (bp1 == 0) {
            if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
            break;
        }
        const int b = bp1 - 1;
        const SampInfo si = load_samp(P, b);
        const int n = min(kTaskBatch, P.nsub - c0);
        for (int j0 = 0; j0 < n; j0 += kIssueGroup) {
            const int nn = min(kIssueGroup, n - j0);
            const uint32_t k0 = group_begin(sh, nn, lane);
            if (k0 == ~0u) {
                if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
                if (lane == 0) producer_done(P, sh);
                return;
            }
            if (lane >= j0 && lane < j0 + nn) {
                const int c = c0 + lane;
                const uint32_t e0 = (uint32_t)c * (uint32_t)ce4;
                const uint32_t bytes = min((uint32_t)ce4, (uint32_t)P.V - e0) * (uint32_t)esz;
                const int s = (int)((k0 + (uint32_t)(lane - j0)) % kFStages);
                Desc d;
                d.kind = kKindSample; d.b = b; d.slot = si.mode; d.c = c;
                d.nvec = (int)(bytes / 16); d.cval = 0.f; d.greedy = 0; d.pad = 0;
                sh.desc[s] = d;
                uint64_t *fb = reinterpret_cast<uint64_t *>(&sh.full[s]);
                mbar_expect_tx(fb, si.mode == 1 ? 2u * bytes : bytes);
                bulk_g2s(sh.buf[s], row_ptr(P, b, si.slot_t, esz) + (size_t)e0 * esz, bytes, fb);
                if (si.mode == 1)
                    bulk_g2s(sh.buf[s] + kSubBytes / 16,
                             row_ptr(P, b, si.slot_d, esz) + (size_t)e0 * esz, bytes, fb);
            }
            group_end(sh, lane);
        }
    }
    if (lane == 0) producer_done(P, sh);
}

// ------------------------------------------------------------------ consumers

// Completion counts a consumer warp has not published yet: finished stream
// items of one row, finished sampler tasks of one request.  Counts are
// published (GPU fence + atomic add) when the warp moves to another row or
// request and before it blocks on a stage that is not ready, so a count never
// waits on a warp that is itself waiting.
struct Pending {
    int row, cnt;   // stream items of row (b * nslot + slot)
    int req, scnt;  // sampler tasks of request b
};

template <int DT>
__device__ void flush_rows(const Params &P, Pending &pd, int lane) {
    if (pd.cnt == 0) return;
    const int row = pd.row, cnt = pd.cnt;
    pd.cnt = 0;
    int last = 0;
    if (lane == 0) {
        __threadfence();
        last = atomicAdd(&P.row_cnt[row], cnt) + cnt == P.nchunk8;
    }
    if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
    __threadfence();
    const int b = row / P.nslot, slot = row - b * P.nslot;
    const ReqInfo rq = P.req[b];
    const float4 rsv = combine_row(P, b, slot, rq.greedy != 0, rq.c, lane);
    const int nrows = rq.greedy ? rq.L + 1 : 2 * rq.L + 1;
    if (lane == 0) {
        P.rowstat[row] = rsv;
        __threadfence();
        last = atomicAdd(&P.req_cnt[b], 1) == nrows - 1;
    }
    if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
    __threadfence();
    decide_request<DT>(P, b, lane);
}

template <int DT>
__device__ void flush_samples(const Params &P, Pending &pd, int lane) {
    if (pd.scnt == 0) return;
    const int b = pd.req, cnt = pd.scnt;
    pd.scnt = 0;
    int last = 0;
    if (lane == 0) {
        __threadfence();
        last = atomicAdd(&P.samp_cnt[b], cnt) + cnt == P.nsub;
    }
    if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
    __threadfence();
    find_request<DT>(P, b, lane);
}

template <int DT>
__device__ void consumer_loop(const Params &P, FusedShared &sh, int cw, int lane) {
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE8 = kStageBytes / ESZ;
    Pending pd{-1, 0, -1, 0};
    for (uint32_t k = (uint32_t)cw;; k += (uint32_t)kFC) {
        const int s = (int)(k % kFStages);
        uint64_t *fb = reinterpret_cast<uint64_t *>(&sh.full[s]);
        const uint32_t par = (k / kFStages) & 1u;
        int ready = 0;
        if (lane == 0) ready = mbar_try_wait(fb, par);
        if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) {
            flush_rows<DT>(P, pd, lane);
            flush_samples<DT>(P, pd, lane);
            if (!mbar_wait_bounded(fb, par, kWaitLimitNs)) {
                if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
                return;
            }
        } else {
            mbar_wait_bounded(fb, par, kWaitLimitNs);  // completes at once: every lane observes it
        }
        const Desc d = sh.desc[s];
        if (d.kind == kKindEnd) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[s]);
            flush_rows<DT>(P, pd, lane);
            flush_samples<DT>(P, pd, lane);
            return;
        }
        if (d.kind == kKindStream) {
            flush_samples<DT>(P, pd, lane);  // publish finished sampler tasks at once
            uint4 v[kStreamVec];
#pragma unroll
            for (int i = 0; i < kStreamVec; ++i) v[i] = sh.buf[s][i * 32 + lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[s]);
            const float4 part = stream_partial<DT>(v, d.nvec, d.greedy != 0, d.cval, d.c * CE8, lane);
            const int row = d.b * P.nslot + d.slot;
            if (lane == 0) P.part[(size_t)row * P.nchunk8 + d.c] = part;
            if (row != pd.row) {
                flush_rows<DT>(P, pd, lane);
                pd.row = row;
            }
            ++pd.cnt;
        } else {
            uint4 vt[kSubVec], vd[kSubVec];
            const uint32_t ni = Fmt<DT>::kNegInfWord;
            const bool resid = d.slot == 1;
#pragma unroll
            for (int i = 0; i < kSubVec; ++i) {
                vt[i] = sh.buf[s][i * 32 + lane];
                vd[i] = resid ? sh.buf[s][kSubBytes / 16 + i * 32 + lane] : make_uint4(ni, ni, ni, ni);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[s]);
            flush_rows<DT>(P, pd, lane);  // publish finished rows at once
            const SampInfo si = load_samp(P, d.b);
            float A, Bs, W;
            FF st, sd;
            sample_masses<DT>(vt, vd, d.nvec, si, A, Bs, W, st, sd, lane);
            if (lane == 0) {
                P.sub[(size_t)d.b * P.nsub + d.c] = make_float4(A, Bs, W, 0.f);
                P.sexact[(size_t)d.b * P.nsub + d.c] = make_float4(st.hi, st.lo, sd.hi, sd.lo);
            }
            if (d.b != pd.req) {
                flush_samples<DT>(P, pd, lane);
                pd.req = d.b;
            }
            ++pd.scnt;
        }
    }
}

// ------------------------------------------------------------------ the kernel

template <int DT>
__global__ void __launch_bounds__(kFThreads, 3) sv_fused(Params P) {
    constexpr int ESZ = Fmt<DT>::kESZ;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kFStages; ++s) {
            mbar_init(reinterpret_cast<uint64_t *>(&sh.full[s]), 1);
            mbar_init(reinterpret_cast<uint64_t *>(&sh.empty[s]), 1);
        }
        sh.prod_seq = 0u;
        sh.prod_done = 0u;
        sh.prod_lock = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the outputs of sv_prep (row list, counters) are read below
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        stream_producer<DT>(P, sh, lane);
        return;
    }
    if (warp == 1) {
        task_producer(P, sh, ESZ, lane);
        return;
    }

    // -------------------------------------------------------------- consumers
    consumer_loop<DT>(P, sh, warp - kFProd, lane);
}

} // namespace sv
