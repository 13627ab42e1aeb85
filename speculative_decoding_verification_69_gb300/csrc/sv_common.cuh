// sv_common.cuh -- device building blocks shared by the verification kernels:
// element access for bf16 / fp32 logit vectors, packed f32x2 arithmetic,
// two-float (double-single) sums, warp / CTA reductions, bulk-copy and
// mbarrier primitives with bounded waits, and Philox4x32-10.
//
// Numerics contract.
//   * The streaming statistics pass needs only float accuracy (~1e-7): per
//     chunk the exact max m_c and s_c = sum_v 2^((z_v - m_c) * c), c = log2(e)/T
//     as a float, formed as ex2.approx((z - m_c) * c) and summed in float.
//   * The sampler re-forms the weights of the one row (pair) it draws from with
//     the row max m and a two-float c = c_hi + c_lo:
//         e_v = ex2.approx(fma(d, c_hi, d * c_lo)),  d = z_v - m,
//     and sums them exactly (Fast2Sum against a biased accumulator), so its
//     normaliser carries no coherent error; every kernel that re-forms e_v uses
//     the same explicitly rounded intrinsics, so the values agree bit for bit.
//   * c_hi is rounded toward zero and c_lo >= FLT_MIN > 0, so d = -inf gives
//     -inf (weight 0), never NaN.
#pragma once
#include <cstdint>
#include <cfloat>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace sv {

constexpr int kThreads = 256;   // threads per CTA of the per-request kernels
constexpr int kWarps = kThreads / 32;
constexpr int kChunkBytes = 4096;                 // logits one warp handles per item
constexpr int kVecPerLane = kChunkBytes / 16 / 32; // 16-byte vectors per lane per item

enum { kF32 = 0, kBF16 = 1 };

template <int DT> struct Fmt;
template <> struct Fmt<kBF16> {
    static constexpr int kEPV = 8;  // elements per 16-byte vector
    static constexpr int kESZ = 2;
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
};
template <> struct Fmt<kF32> {
    static constexpr int kEPV = 4;
    static constexpr int kESZ = 4;
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
};

template <int DT> __host__ __device__ constexpr int chunk_elems() {
    return kChunkBytes / Fmt<DT>::kESZ;
}

// ------------------------------------------------------------------ loads

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// One 16-byte vector of elements [e0, e0+EPV) of a row; elements at or past V
// read as -inf.  VEC: the row is 16-byte aligned and V is a multiple of EPV.
template <int DT, bool VEC>
__device__ __forceinline__ uint4 load_vec(const char *row, long long e0, int V) {
    constexpr int EPV = Fmt<DT>::kEPV;
    const uint32_t ni = Fmt<DT>::kNegInfWord;
    if (VEC) {
        if (e0 < V) return ld_stream_v4(row + e0 * Fmt<DT>::kESZ);
        return make_uint4(ni, ni, ni, ni);
    } else {
        uint32_t w[4] = {ni, ni, ni, ni};
        if (DT == kBF16) {
            const uint16_t *r = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
            for (int i = 0; i < EPV; ++i) {
                long long e = e0 + i;
                uint32_t h = e < V ? (uint32_t)__ldg(r + e) : 0xFF80u;
                if (i & 1) w[i >> 1] = (w[i >> 1] & 0x0000FFFFu) | (h << 16);
                else w[i >> 1] = (w[i >> 1] & 0xFFFF0000u) | h;
            }
        } else {
            const uint32_t *r = reinterpret_cast<const uint32_t *>(row);
#pragma unroll
            for (int i = 0; i < EPV; ++i) {
                long long e = e0 + i;
                w[i] = e < V ? __ldg(r + e) : ni;
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Element i of a vector as float (exact).
template <int DT> __device__ __forceinline__ float elem(const uint4 &v, int i) {
    const uint32_t *w = &v.x;
    if (DT == kBF16) {
        uint32_t x = w[i >> 1];
        return __uint_as_float((i & 1) ? (x & 0xFFFF0000u) : (x << 16));
    } else {
        return __uint_as_float(w[i]);
    }
}

// Maximum element of a vector (exact).
template <int DT> __device__ __forceinline__ float vec_max(const uint4 &v) {
    if (DT == kBF16) {
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
        __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162 *>(&v.z);
        __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162 *>(&v.w);
        __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        return fmaxf(__low2float(m), __high2float(m));
    } else {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}

// ------------------------------------------------------------------ f32x2

__device__ __forceinline__ unsigned long long f2u(float2 a) {
    return *reinterpret_cast<unsigned long long *>(&a);
}
__device__ __forceinline__ float2 u2f(unsigned long long a) {
    return *reinterpret_cast<float2 *>(&a);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
    return u2f(d);
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Scaled weights of an element pair: 2^((z - m) * c + l), c = c_hi + c_lo.
__device__ __forceinline__ float2 weight2l(float2 z, float2 m2, float2 chi2, float2 clo2, float2 l2) {
    float2 d = sub2(z, m2);
    float2 t = fma2(d, chi2, fma2(d, clo2, l2));
    return make_float2(ex2(t.x), ex2(t.y));
}

// ------------------------------------------------------------------ two-float

struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_add(FF a, FF b) {
    float s = __fadd_rn(a.hi, b.hi);
    float bb = __fsub_rn(s, a.hi);
    float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    float hi = __fadd_rn(s, e);
    float lo = __fsub_rn(e, __fsub_rn(hi, s));
    return FF{hi, lo};
}

// a + b as an unevaluated two-float sum (Knuth's TwoSum: no ordering needed).
__device__ __forceinline__ FF two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return FF{s, e};
}

__device__ __forceinline__ FF ff_shfl_xor(FF a, int m) {
    return FF{__shfl_xor_sync(0xFFFFFFFFu, a.hi, m), __shfl_xor_sync(0xFFFFFFFFu, a.lo, m)};
}

__device__ __forceinline__ double ff_to_double(FF a) { return (double)a.hi + (double)a.lo; }

// Per-thread accumulator of non-negative terms <= bias: Fast2Sum against a
// biased high part keeps every rounding error exactly in the low part.
struct BiasAcc2 {
    float2 h, l;
    float bias;
    __device__ __forceinline__ void init(float b) {
        bias = b;
        h = make_float2(b, b);
        l = make_float2(0.f, 0.f);
    }
    __device__ __forceinline__ void add(float2 e) {
        float2 s = add2(h, e);
        float2 z = sub2(s, h);
        float2 err = sub2(e, z);
        l = add2(l, err);
        h = s;
    }
    __device__ __forceinline__ FF total() const {
        FF a{__fsub_rn(h.x, bias), l.x};
        FF b{__fsub_rn(h.y, bias), l.y};
        return ff_add(a, b);
    }
};

// ------------------------------------------------------------------ warp reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ FF warp_sum_ff(FF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff_shfl_xor(v, o));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ------------------------------------------------------------------ bulk copies

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier shared-memory accesses before later bulk
// (async-proxy) writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of `bar`, giving up after `limit_ns` nanoseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------------ packed helpers

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Programmatic dependent launch: wait for the previous kernel's results /
// allow the next kernel to be scheduled.  No-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// ------------------------------------------------------------------ Philox4x32-10

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): each round
// multiplies words 0 and 2 by the two round constants, swaps and xors the
// high halves with the other words and the key; the key advances by the two
// Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a = c.x, b = c.z;
        const uint32_t hi_a = __umulhi(0xD2511F53u, a), lo_a = 0xD2511F53u * a;
        const uint32_t hi_b = __umulhi(0xCD9E8D57u, b), lo_b = 0xCD9E8D57u * b;
        c = make_uint4(hi_b ^ c.y ^ k0, lo_b, hi_a ^ c.w ^ k1, lo_a);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Acceptance uniform (draw 0): the top 24 bits of word 0 -> [0,1), a float
// (24 bits, so exact).
__device__ __forceinline__ float uniform_accept_f(unsigned long long seed, uint32_t b, uint32_t k) {
    uint4 w = philox4x32_10(make_uint4(b, k, 0u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32));
    return (float)(w.x >> 8) * 0x1p-24f;
}

// Sampling uniform (draw 1): 53 bits of (w0:w1) -> [0,1).
__device__ __forceinline__ double uniform_sample(unsigned long long seed, uint32_t b, uint32_t k) {
    uint4 w = philox4x32_10(make_uint4(b, k, 1u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32));
    unsigned long long v = ((unsigned long long)w.x << 32) | (unsigned long long)w.y;
    return (double)(v >> 11) * 0x1p-53;
}

} // namespace sv
