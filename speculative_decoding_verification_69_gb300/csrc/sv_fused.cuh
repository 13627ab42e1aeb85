// sv_fused.cuh -- the fused, persistent verification kernel (16-byte aligned rows).
//
// One launch streams every needed logit row once and finishes every request
// inside the same grid, so the row (pair) a rejected request samples from is
// re-read while it is still resident in L2.  Every warp works on its own:
//
//   * stream items (4 KiB of one needed row) are claimed in small batches from a
//     global counter; the batch's row metadata is gathered across the lanes and
//     each item is bulk-copied into the warp's own ring of kRing stages of
//     shared memory, refilled as soon as a stage has been read into registers;
//   * per item the warp computes a chunk partial (max and either the lowest
//     argmax or the sum of 2^((z - max) log2(e)/T)); the last chunk of a row
//     combines the row, the last row of a request decides it (acceptance rule,
//     first rejection, outputs) and publishes its sampler tasks;
//   * sampler tasks (4 KiB chunks of the row, or row pair, to draw from) are
//     claimed by compare-and-swap only once published, read with plain loads
//     (the rows are still in L2) and reduced to exact residual / target masses;
//     the last task of a request draws the token (inverse CDF).
//
// Completion counts are published (GPU fence + atomic add) when a warp moves
// to another row or request and before it waits for other warps' work (task
// publication), so no count is held by a warp that waits on it.  Work is claimed, never owned in advance: CTAs that are not
// resident hold no work.  Every wait is bounded (SPEC_DEV_TIMEOUT on expiry).
#pragma once
#include "sv_common.cuh"

namespace sv {

constexpr int kFWarps = 8;                     // warps per CTA
constexpr int kFThreads = kFWarps * 32;
constexpr int kRing = 3;                       // bulk-copy stages per warp
constexpr int kStageBytes = 4096;              // one stream item
constexpr int kStreamVec = kStageBytes / 16 / 32;  // 8 vectors per lane
constexpr int kSubBytes = 4096;                // per row of a sampler task
constexpr int kSubVec = kSubBytes / 16 / 32;   // 8 vectors per lane
constexpr int kStreamBatch = 32;               // stream items per claim (one per lane)
constexpr int kTaskClaim = 2;                  // sampler tasks per claim

enum { kKindStream = 0, kKindSample = 1, kKindEnd = 2 };

struct Desc {
    int kind, b, slot, c;
    int nvec;     // valid 16-byte vectors of the (first) row
    float cval;   // log2(e)/T as float (stream items)
    int greedy;
    int pad;
};

// One warp's ring.  Item k (the warp's k-th issued item) uses stage k % kRing
// and phase (k / kRing) & 1 of its barrier: one warp issues and consumes in
// order, so a waiter is never more than one phase away.
struct WarpRing {
    uint4 buf[kRing][kStageBytes / 16];
    Desc desc[kRing];
    Desc meta[kStreamBatch];      // the claimed batch, one entry per lane
    unsigned long long full[kRing];
};

struct FusedShared {
    WarpRing ring[kFWarps];
};

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Atomic add with release semantics: this thread's earlier stores are visible
// before the add; the result is only needed later, so the warp keeps going.
__device__ __forceinline__ int atom_add_release(int *p, int v) {
    int old;
    asm volatile("atom.add.release.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
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
// vector i*32 + lane of the chunk): greedy rows {max, -, lowest argmax, -},
// sampled rows {max, sum 2^((z - max) c), -1, -}; the caller stores the call's
// epoch in .w.
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
        return make_float4(m, 0.f, __int_as_float(warp_min_int(idx)), 0.f);
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
    return make_float4(m, warp_sum(s), __int_as_float(-1), 0.f);
}

// ------------------------------------------------------------------ row combine

// Row statistics from its chunk partials (one warp): {max, S (sampled) or 0,
// lowest argmax (greedy) as int bits, -}.
constexpr int kPerLane = 4;  // chunk records held in registers per lane (128 per warp)

// A chunk partial of this call: its .w holds the call's epoch.  Partials are
// published with relaxed counters, so the combining warp re-reads (bounded) a
// record until its tag shows it; a 16-byte record is written in one store.
__device__ __forceinline__ float4 load_partial(const float4 *p, unsigned int epoch, bool &ok) {
    float4 q = __ldcg(p);
    if (__float_as_uint(q.w) == epoch) return q;
    const unsigned long long t0 = global_ns();
    for (;;) {
        __nanosleep(32);
        q = __ldcg(p);
        if (__float_as_uint(q.w) == epoch) return q;
        if (global_ns() - t0 > kWaitLimitNs) {
            ok = false;
            return q;
        }
    }
}

__device__ __forceinline__ float4 combine_row(const Params &P, int b, int slot, bool greedy,
                                              float c, int lane) {
    const float4 *pp = P.part + ((size_t)b * P.nslot + slot) * P.nchunk8;
    const int n = P.nchunk8;
    float m = -INFINITY, S = 0.f;
    int amax = INT_MAX;
    bool ok = true;
    // all loads of a round are issued before any is used
    for (int base = 0; base < n; base += 32 * kPerLane) {
        float4 q[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int ci = base + i * 32 + lane;
            q[i] = ci < n ? __ldcg(&pp[ci]) : make_float4(-INFINITY, 0.f, __int_as_float(INT_MAX), 0.f);
        }
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int ci = base + i * 32 + lane;
            if (ci < n && __float_as_uint(q[i].w) != P.epoch) q[i] = load_partial(&pp[ci], P.epoch, ok);
        }
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
    if (__any_sync(0xFFFFFFFFu, !ok) && lane == 0 && P.dev_status)
        atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
    if (greedy) return make_float4(m, 0.f, __int_as_float(amax), 0.f);
    return make_float4(m, S, __int_as_float(-1), 0.f);
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
            const int e = atomicAdd(P.q_alloc, 1);
            fence_acq_rel_gpu();  // the sampler state is visible before the entry
            *reinterpret_cast<volatile int *>(&P.q_entries[e]) = b + 1;
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
    // each lane owns a contiguous block of chunks; records are loaded at once
    const int per = (nch + 31) / 32;
    const int c0 = lane * per, c1 = min(nch, c0 + per);
    float4 q[kPerLane], e[kPerLane];
    const bool held = per <= kPerLane;
    double st = 0.0, sd = 0.0;
    if (held) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int c = c0 + i;
            q[i] = c < c1 ? __ldcg(&sub[c]) : make_float4(0.f, 0.f, 0.f, 0.f);
            e[i] = c < c1 ? __ldcg(&sex[c]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            st += (double)e[i].x + (double)e[i].y;
            sd += (double)e[i].z + (double)e[i].w;
        }
    } else {
        for (int c = c0; c < c1; ++c) {
            const float4 x = __ldcg(&sex[c]);
            st += (double)x.x + (double)x.y;
            sd += (double)x.z + (double)x.w;
        }
    }
    st = warp_sum_d(st);
    sd = warp_sum_d(sd);
    const double kt = resid ? 1.0 / ((double)si.rho_t * st) : 1.0;
    const double kd = resid ? 1.0 / ((double)si.rho_d * sd) : 0.0;
    auto mass_r = [&](const float4 &x) {
        return resid ? fmax(0.0, kt * (double)x.x - kd * (double)x.y) : (double)x.z;
    };
    double zr = 0.0, zw = 0.0;
    if (held) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            if (c0 + i < c1) {
                zr += mass_r(q[i]);
                zw += (double)q[i].z;
            }
    } else {
        for (int c = c0; c < c1; ++c) {
            const float4 x = __ldcg(&sub[c]);
            zr += mass_r(x);
            zw += (double)x.z;
        }
    }
    const double Zr = warp_sum_d(zr), Zw = warp_sum_d(zw);
    const bool use_w = !resid || !(Zr > 0.0);
    const double theta = si.u * (use_w ? Zw : Zr);
    const double mine = use_w ? zw : zr;
    double incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    double base = incl - mine;
    int my_c = INT_MAX, my_last = -1;
    double my_base = 0.0;
    const bool mine_crosses = base <= theta && base + mine > theta;
    for (int c = c0; c < c1; ++c) {
        const float4 x = held ? q[(c - c0) & (kPerLane - 1)] : __ldcg(&sub[c]);
        const double v = use_w ? (double)x.z : mass_r(x);
        if (v > 0.0) my_last = c;
        if (mine_crosses && my_c == INT_MAX) {
            if (base + v > theta) {
                my_c = c;
                my_base = base;
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
        int last = my_last;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xFFFFFFFFu, last, o));
        ch = last >= 0 ? last : nch - 1;
        th_local = INFINITY;
    }
    // the chosen chunk: all vectors loaded at once, then scanned in order
    const char *rowt = row_ptr(P, b, si.slot_t, ESZ);
    const char *rowd = resid ? row_ptr(P, b, si.slot_d, ESZ) : rowt;
    const long long e0 = (long long)ch * CE;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    const bool two = resid && !use_w;
    uint4 vt[kSubVec], vd[kSubVec];
#pragma unroll
    for (int i = 0; i < kSubVec; ++i) {
        const long long q0 = e0 + (long long)(i * 32 + lane) * EPV;
        vt[i] = load_vec<DT, true>(rowt, q0, P.V);
        vd[i] = two ? load_vec<DT, true>(rowd, q0, P.V) : make_uint4(ni, ni, ni, ni);
    }
    const float2 m2 = make_float2(si.m_t, si.m_d);
    const float2 chi2 = make_float2(si.c_hi, si.c_hi), clo2 = make_float2(si.c_lo, si.c_lo);
    const float2 rho2 = two ? make_float2(si.rho_t, si.rho_d) : make_float2(si.rho_t, 0.f);
    const float dkt = (float)(kt - 1.0), dkd = (float)(kd - 1.0);
    double run = 0.0;
    int found = INT_MAX, last_pos = -1;
#pragma unroll
    for (int i = 0; i < kSubVec; ++i) {
        if (found != INT_MAX) break;
        const long long q0 = e0 + (long long)(i * 32 + lane) * EPV;
        float w[EPV];
#pragma unroll
        for (int k = 0; k < EPV; ++k) {
            const float2 ee = weight2(make_float2(elem<DT>(vt[i], k), elem<DT>(vd[i], k)), m2, chi2, clo2);
            const float2 ab = mul2(ee, rho2);
            float wv;
            if (use_w) wv = ab.x;
            else wv = ab.x > ab.y ? fmaxf(__fsub_rn(__fmaf_rn(ab.x, dkt, ab.x), __fmaf_rn(ab.y, dkd, ab.y)), 0.f) : 0.f;
            w[k] = wv;
            if (wv > 0.f && q0 + k < P.V) last_pos = (int)(q0 + k);
        }
        float vs = w[0];
#pragma unroll
        for (int k = 1; k < EPV; ++k) vs = __fadd_rn(vs, w[k]);
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
            for (int k = 0; k < EPV; ++k) {
                ps = k == 0 ? w[0] : __fadd_rn(ps, w[k]);
                if (tok == INT_MAX && lo_edge + (double)ps > th_local) tok = (int)(q0 + k);
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

// ------------------------------------------------------------------ completion counts

// Completion counts a warp has not published yet: finished stream items of one
// row, finished sampler tasks of one request.
struct Pending {
    int row, cnt;   // stream items of row (b * nslot + slot)
    int req, scnt;  // sampler tasks of request b
    // a posted row count whose result (the counter's previous value, lane 0)
    // is examined at the next flush point
    int post_row, post_cnt, post_old;
};

template <int DT>
__device__ __noinline__ void row_complete(const Params &P, int row, int lane);

// Examine the posted count: if it completed its row, finish the row.
template <int DT>
__device__ __forceinline__ void resolve_rows(const Params &P, Pending &pd, int lane) {
    if (pd.post_cnt == 0) return;
    const int last = __shfl_sync(0xFFFFFFFFu, pd.post_old + pd.post_cnt == P.nchunk8, 0);
    const int row = pd.post_row;
    pd.post_cnt = 0;
    if (last) row_complete<DT>(P, row, lane);
}

// Publish the pending count of the current row (relaxed add: the combining
// warp validates the partials' tags; the result is examined at the next flush
// point or by resolve_rows, so the warp does not wait for it).
template <int DT>
__device__ __forceinline__ void flush_rows(const Params &P, Pending &pd, int lane) {
    resolve_rows<DT>(P, pd, lane);
    if (pd.cnt == 0) return;
    int old = 0;
    if (lane == 0) old = atomicAdd(&P.row_cnt[pd.row], pd.cnt);  // partials carry tags: relaxed
    pd.post_row = pd.row;
    pd.post_cnt = pd.cnt;
    pd.post_old = old;
    pd.cnt = 0;
}

// The last chunk of a row: combine the row, and decide the request if this was
// its last row.
template <int DT>
__device__ __noinline__ void row_complete(const Params &P, int row, int lane) {
    int last = 0;
    fence_acq_rel_gpu();
    const int b = row / P.nslot, slot = row - b * P.nslot;
    const ReqInfo rq = P.req[b];
    const float4 rsv = combine_row(P, b, slot, rq.greedy != 0, rq.c, lane);
    const int nrows = rq.greedy ? rq.L + 1 : 2 * rq.L + 1;
    if (lane == 0) {
        P.rowstat[row] = rsv;
        last = atom_add_release(&P.req_cnt[b], 1) == nrows - 1;
    }
    if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
    fence_acq_rel_gpu();
    decide_request<DT>(P, b, lane);
}

template <int DT>
__device__ void flush_samples(const Params &P, Pending &pd, int lane) {
    if (pd.scnt == 0) return;
    const int b = pd.req, cnt = pd.scnt;
    pd.scnt = 0;
    int last = 0;
    if (lane == 0) last = atom_add_release(&P.samp_cnt[b], cnt) + cnt == P.nsub;
    if (!__shfl_sync(0xFFFFFFFFu, last, 0)) return;
    fence_acq_rel_gpu();
    find_request<DT>(P, b, lane);
}

// ------------------------------------------------------------------ sampler tasks

// Request entry e (publication order) owns task indices [e * nsub_pad,
// (e + 1) * nsub_pad), nsub_pad = nsub rounded up to kTaskClaim.
//
// While streaming, a warp takes tasks only if they are already published
// (compare-and-swap, at most two tries per stream batch), so a claim never
// stops it.  Returns the first claimed task index, or ~0ull.
__device__ __forceinline__ unsigned long long claim_published(const Params &P,
                                                              unsigned long long total,
                                                              unsigned long long nsub_pad, int lane) {
    unsigned long long got = ~0ull;
    if (lane == 0) {
        unsigned long long h = *reinterpret_cast<volatile unsigned long long *>(P.q_head);
        for (int tries = 0; tries < 2 && h < total; ++tries) {
            if (ld_volatile_int(&P.q_entries[h / nsub_pad]) == 0) break;
            const unsigned long long old = atomicCAS(P.q_head, h, h + kTaskClaim);
            if (old == h) {
                got = h;
                break;
            }
            h = old;
        }
        if (got != ~0ull) __threadfence();
    }
    return __shfl_sync(0xFFFFFFFFu, got, 0);
}

// After streaming, a warp claims the next tasks with one atomic add and waits
// (bounded) until their request is published; it has nothing else to do, and
// publication depends only on stream items other warps already hold.
// Returns the first claimed task index, ~0ull when all are claimed, or ~1ull
// on timeout.
__device__ __forceinline__ unsigned long long claim_next(const Params &P, unsigned long long total,
                                                         unsigned long long nsub_pad, int lane) {
    unsigned long long got = ~0ull;
    if (lane == 0) {
        const unsigned long long h = atomicAdd(P.q_head, (unsigned long long)kTaskClaim);
        if (h < total) {
            got = h;
            const int *flag = &P.q_entries[h / nsub_pad];
            if (ld_volatile_int(flag) == 0) {
                const unsigned long long t0 = global_ns();
                unsigned int nap = 64;
                while (ld_volatile_int(flag) == 0) {
                    if (global_ns() - t0 > kWaitLimitNs) {
                        got = ~1ull;
                        break;
                    }
                    __nanosleep(nap);
                    if (nap < 1024) nap <<= 1;
                }
            }
            __threadfence();
        }
    }
    return __shfl_sync(0xFFFFFFFFu, got, 0);
}

// Process the (up to kTaskClaim) sampler tasks starting at task index h.
template <int DT>
__device__ void run_tasks(const Params &P, unsigned long long h, unsigned long long nsub_pad,
                          Pending &pd, int lane) {
    constexpr int EPV = Fmt<DT>::kEPV;
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE4 = kSubBytes / ESZ;
    const unsigned long long e = h / nsub_pad;
    const int c0 = (int)(h - e * nsub_pad);
    const int b = ld_volatile_int(&P.q_entries[e]) - 1;
    const SampInfo si = load_samp(P, b);
    const bool resid = si.mode == 1;
    const char *rowt = row_ptr(P, b, si.slot_t, ESZ);
    const char *rowd = resid ? row_ptr(P, b, si.slot_d, ESZ) : rowt;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    if (b != pd.req) {
        flush_samples<DT>(P, pd, lane);
        pd.req = b;
    }
    const int c1 = min(c0 + kTaskClaim, P.nsub);
    for (int c = c0; c < c1; ++c) {
        const long long e0 = (long long)c * CE4;
        const int nvec = (int)((min((long long)CE4, (long long)P.V - e0) + EPV - 1) / EPV);
        uint4 vt[kSubVec], vd[kSubVec];
#pragma unroll
        for (int i = 0; i < kSubVec; ++i) {
            const long long q = e0 + (long long)(i * 32 + lane) * EPV;
            vt[i] = load_vec<DT, true>(rowt, q, P.V);
            vd[i] = resid ? load_vec<DT, true>(rowd, q, P.V) : make_uint4(ni, ni, ni, ni);
        }
        float A, Bs, W;
        FF st, sd;
        sample_masses<DT>(vt, vd, nvec, si, A, Bs, W, st, sd, lane);
        if (lane == 0) {
            P.sub[(size_t)b * P.nsub + c] = make_float4(A, Bs, W, 0.f);
            P.sexact[(size_t)b * P.nsub + c] = make_float4(st.hi, st.lo, sd.hi, sd.lo);
        }
        ++pd.scnt;
    }
}

// ------------------------------------------------------------------ the kernel

template <int DT>
__global__ void __launch_bounds__(kFThreads, 2) sv_fused(Params P) {
    constexpr int ESZ = Fmt<DT>::kESZ;
    constexpr int CE = kStageBytes / ESZ;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FusedShared &sh = *reinterpret_cast<FusedShared *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpRing &rg = sh.ring[warp];
    if (lane == 0) {
        for (int s = 0; s < kRing; ++s) mbar_init(reinterpret_cast<uint64_t *>(&rg.full[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    // the outputs of sv_prep (row list, counters) are read below
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const uint32_t n_stream = (uint32_t)(*P.row_count) * (uint32_t)P.nchunk8;
    const unsigned long long nsub_pad =
        (unsigned long long)((P.nsub + kTaskClaim - 1) / kTaskClaim) * kTaskClaim;
    const unsigned long long total_tasks = (unsigned long long)(*P.n_sampled) * nsub_pad;
    const uint32_t total_warps = gridDim.x * kFWarps;

    Pending pd{-1, 0, -1, 0, -1, 0, 0};
    uint32_t k_iss = 0, k_cons = 0;  // issued / consumed items of this warp
    int bcount = 0, bnext = 0;       // items in the current batch (metadata in rg.meta), next to issue
    bool stream_left = true;
    // the next batch is claimed one batch ahead; lane 0 holds the claim's result
    uint32_t claim = max(1u, min((uint32_t)kStreamBatch, n_stream / (2u * total_warps)));
    uint32_t ahead_base = 0, ahead_claim = claim;
    if (lane == 0) ahead_base = atomicAdd(P.stream_head, claim);
    // task-queue state read one batch ahead (lane 0)
    unsigned long long pf_head = 0;
    int pf_alloc = 0;

    // Switch to the batch claimed ahead and claim the following one.
    auto next_batch = [&]() -> bool {
        const uint32_t base = __shfl_sync(0xFFFFFFFFu, ahead_base, 0);
        if (base >= n_stream) {
            stream_left = false;
            return false;
        }
        bcount = (int)min(ahead_claim, n_stream - base);
        bnext = 0;
        if (lane < bcount) {
            const uint32_t item = base + (uint32_t)lane;
            const uint32_t ri = item / (uint32_t)P.nchunk8;
            const uint32_t c = item - ri * (uint32_t)P.nchunk8;
            const int4 r = P.rows[ri];
            Desc m;
            m.kind = kKindStream; m.b = r.x; m.slot = r.y; m.c = (int)c;
            m.nvec = (int)(min((uint32_t)CE, (uint32_t)P.V - c * CE) * ESZ / 16);
            m.cval = __int_as_float(r.w); m.greedy = r.z; m.pad = 0;
            rg.meta[lane] = m;
        }
        // smaller claims near the end keep the warps' finishing times together
        const uint32_t left = n_stream - base - (uint32_t)bcount;
        claim = max(1u, min((uint32_t)kStreamBatch, left / (2u * total_warps)));
        ahead_claim = claim;
        if (lane == 0) {
            ahead_base = atomicAdd(P.stream_head, claim);
            pf_head = *reinterpret_cast<volatile unsigned long long *>(P.q_head);
            pf_alloc = ld_volatile_int(P.q_alloc);
        }
        __syncwarp();
        return true;
    };

    // Issue the next stream item into stage k_iss % kRing (free by construction).
    auto refill = [&]() -> bool {
        if (bnext == bcount && (!stream_left || !next_batch())) return false;
        const int j = bnext++;
        const int s = (int)(k_iss % kRing);
        if (lane == 0) {
            const Desc m = rg.meta[j];
            const uint32_t bytes = (uint32_t)m.nvec * 16u;
            fence_proxy_async();  // the stage's previous contents were read by this warp
            rg.desc[s] = m;
            uint64_t *fb = reinterpret_cast<uint64_t *>(&rg.full[s]);
            mbar_expect_tx(fb, bytes);
            bulk_g2s(rg.buf[s], row_ptr(P, m.b, m.slot, ESZ) + (size_t)m.c * CE * ESZ, bytes, fb);
        }
        __syncwarp();
        ++k_iss;
        return true;
    };

    for (int i = 0; i < kRing; ++i)
        if (!refill()) break;
    bool failed = false;
    while (k_cons != k_iss) {
        const int s = (int)(k_cons % kRing);
        uint64_t *fb = reinterpret_cast<uint64_t *>(&rg.full[s]);
        const uint32_t par = (k_cons / kRing) & 1u;
        // this wait depends on nothing but the warp's own copies: pending counts may stay pending
        if (!mbar_wait_bounded(fb, par, kWaitLimitNs)) {
            failed = true;
            break;
        }
        const Desc d = rg.desc[s];
        uint4 v[kStreamVec];
#pragma unroll
        for (int i = 0; i < kStreamVec; ++i) v[i] = rg.buf[s][i * 32 + lane];
        __syncwarp();
        ++k_cons;
        // task-queue state prefetched at the previous batch switch
        const int tasks_hint =
            __shfl_sync(0xFFFFFFFFu, (int)(pf_head < (unsigned long long)pf_alloc * nsub_pad), 0);
        const bool switching = bnext == bcount;
        refill();
        float4 part = stream_partial<DT>(v, d.nvec, d.greedy != 0, d.cval, d.c * CE, lane);
        part.w = __uint_as_float(P.epoch);
        const int row = d.b * P.nslot + d.slot;
        if (lane == 0) P.part[(size_t)row * P.nchunk8 + d.c] = part;
        if (row != pd.row) {
            flush_rows<DT>(P, pd, lane);
            pd.row = row;
        }
        ++pd.cnt;
        if (switching && tasks_hint) {
            // published sampler tasks were waiting at the last batch switch: take some
            const unsigned long long h = claim_published(P, total_tasks, nsub_pad, lane);
            if (h != ~0ull) {
                flush_rows<DT>(P, pd, lane);
                resolve_rows<DT>(P, pd, lane);
                run_tasks<DT>(P, h, nsub_pad, pd, lane);
                flush_samples<DT>(P, pd, lane);
            }
        }
    }
    if (failed) {
        if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
        for (uint32_t k = k_cons + 1; k < k_iss; ++k)  // let this warp's copies land
            mbar_wait_bounded(reinterpret_cast<uint64_t *>(&rg.full[k % kRing]), (k / kRing) & 1u,
                              kWaitLimitNs);
        return;
    }
    // stream exhausted: sampler tasks until every task is claimed
    flush_rows<DT>(P, pd, lane);
    resolve_rows<DT>(P, pd, lane);
    for (;;) {
        const unsigned long long h = claim_next(P, total_tasks, nsub_pad, lane);
        if (h == ~0ull) break;
        if (h == ~1ull) {
            if (lane == 0 && P.dev_status) atomicOr(P.dev_status, SPEC_DEV_TIMEOUT);
            break;
        }
        run_tasks<DT>(P, h, nsub_pad, pd, lane);
        flush_samples<DT>(P, pd, lane);
    }
    flush_samples<DT>(P, pd, lane);
}

} // namespace sv
