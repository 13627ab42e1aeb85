// lm_gemm.cuh -- the LM-head product z = H W^T on the sm_103a tensor cores,
// with the logits consumed in the epilogue (never stored in full).
//
// Shapes: H [M, d] bf16 row-major (one hidden state per logit row), W [V, d]
// bf16 row-major (one vocabulary entry per row, K-major for the product), d a
// multiple of 64.  A CTA owns a 128 x 256 tile of z (128 rows, 256 vocabulary
// entries) at a time and walks the tiles of the grid persistently, vocabulary
// block major (consecutive tiles share one W tile, so W streams from HBM once
// while H stays in L2).
//
// Per CTA (one per SM, 192 threads):
//   warp 0      TMA producer: per 64-wide k block one 128 x 64 tile of H and
//               one 256 x 64 tile of W into a 4-stage shared-memory ring
//               (128-byte swizzle, the layout the MMA descriptors name);
//   warp 1      allocates the 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and, from one thread, issues the tcgen05.mma
//               (kind::f16, M = 128, N = 256, K = 16, fp32 accumulate) of each
//               stage, releasing the stage with tcgen05.commit;
//   warps 2-5   epilogue: each thread owns one row of the finished tile and
//               reads its 256 accumulators from TMEM (tcgen05.ld, 32 columns at
//               a time); what it does with them is the Epi functor's business.
// The two accumulators alternate, so the epilogue of a tile overlaps the MMAs
// of the next one.
//
// Every wait is bounded: a barrier that stays incomplete for kLmWaitNs sets
// the CTA's abort flag and SPEC_DEV_TIMEOUT; all roles then leave their loops,
// the producer waits (bounded) for its copies in flight, the MMA thread for its
// MMAs, and the TMEM is freed before the CTA exits.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "sv_common.cuh"

namespace sv {

constexpr int kLmBM = 128;        // rows of a tile (MMA M, TMEM lanes)
constexpr int kLmBN = 256;        // vocabulary entries of a tile (MMA N, TMEM columns)
constexpr int kLmBK = 64;         // k block: one 128-byte swizzle atom of bf16
constexpr int kLmStages = 4;
constexpr int kLmThreads = 192;
constexpr uint32_t kLmBytesA = kLmBM * kLmBK * 2;  // 16 KiB
constexpr uint32_t kLmBytesB = kLmBN * kLmBK * 2;  // 32 KiB
constexpr uint32_t kLmTmemCols = 2 * kLmBN;        // two fp32 accumulators
constexpr unsigned long long kLmWaitNs = 4000000000ull;  // 4 s

struct LmShared {
    uint8_t a[kLmStages][kLmBytesA];  // each 1024-byte aligned (swizzle atoms)
    uint8_t b[kLmStages][kLmBytesB];
    uint64_t full[kLmStages], empty[kLmStages];
    uint64_t acc_full[2], acc_empty[2], done;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kLmSmem = sizeof(LmShared) + 1024;  // room to align the base to 1024

// ------------------------------------------------------------------ PTX wrappers

// 2D tiled TMA load of the box at (x = k offset in elements, y = row) into
// shared memory; completion as transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart
// (stride byte offset), leading byte offset unused for this layout, descriptor
// version 1 (bits 46-48), swizzle mode 2 = 128 bytes (bits 61-63).  The k step
// inside the atom advances the start address by 32 bytes per 16 elements.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kLmIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                              ((uint32_t)(kLmBN >> 3) << 17) | ((uint32_t)(kLmBM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kLmIdesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane (shape
// 32x32b: lane i of the warp reads TMEM lane base + i), waited for in the same
// statement so no use can be scheduled before the data arrive.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait (limit_ns) that also gives up as soon as another role of the
// CTA has.
__device__ __forceinline__ bool lm_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                        unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ the kernel

// The rows come in two segments with their own tensor maps: rows [0, M0) of
// tmA0, then rows [0, M1) of tmA1 (M1 = 0: one segment), each cut into row
// tiles of its own.  M0 = min(M0, mult * *M_dev) when M_dev is given (a count
// only the device knows).  Epi::row(seg, r, valid, n0, V, taddr) is called by
// every epilogue thread for each finished tile, convergently per warp
// (tcgen05.ld is warp-collective): row r of segment seg (valid = r below the
// segment's row count), the tile's first vocabulary entry n0, and the TMEM
// address of the row's 256 fp32 accumulators (column j at taddr + j).
// Columns at or past V and rows past the segment's count hold zeros (the TMA
// fills them): Epi masks them.  diag (diagnostics only): the producer issues
// no copy, so the first wait on a stage runs out after diag_ns and the CTA
// gives up as on a real timeout.
template <class Epi>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
            const __grid_constant__ CUtensorMap tmB, int M0, int M1, const int *M_dev, int mult,
            int V, int d, Epi epi, uint32_t *status, int diag, unsigned long long diag_ns) {
    const unsigned long long limit_ns = diag ? diag_ns : kLmWaitNs;
    extern __shared__ uint8_t lm_raw[];
    LmShared &sh = *reinterpret_cast<LmShared *>((reinterpret_cast<uintptr_t>(lm_raw) + 1023) &
                                                  ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kLmStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh.acc_full[i], 1);
            mbar_init(&sh.acc_empty[i], 4);  // one arrival per epilogue warp
        }
        mbar_init(&sh.done, 1);
        sh.abort = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmA0);
        if (M1 > 0) tma_prefetch_map(&tmA1);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kLmTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // a device-side row count comes from the previous kernel
    const uint32_t tmem = sh.tmem_base;
    if (M_dev) M0 = min(M0, mult * *M_dev);
    const int mt0 = (M0 + kLmBM - 1) / kLmBM;
    const int m_tiles = mt0 + (M1 + kLmBM - 1) / kLmBM;
    const int n_tiles = (V + kLmBN - 1) / kLmBN;
    const int k_blocks = d / kLmBK;
    const int num_tiles = m_tiles * n_tiles;
    volatile int *abort = &sh.abort;

    if (warp == 0) {
        if (lane == 0) {  // ---------------------------------------- TMA producer
            uint32_t it = 0;
            for (int tile = blockIdx.x; tile < num_tiles && !*abort; tile += gridDim.x) {
                const int m_blk = tile % m_tiles, n_blk = tile / m_tiles;
                const bool seg1 = m_blk >= mt0;
                const CUtensorMap *ta = seg1 ? &tmA1 : &tmA0;
                const int row0 = (seg1 ? m_blk - mt0 : m_blk) * kLmBM;
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const int s = (int)(it % kLmStages);
                    const uint32_t fill = it / kLmStages;
                    if (fill > 0 && !lm_wait(&sh.empty[s], (fill - 1) & 1u, abort, limit_ns)) break;
                    if (diag) break;  // nothing is copied: the consumers' waits run out
                    mbar_expect_tx(&sh.full[s], kLmBytesA + kLmBytesB);
                    tma_load_2d(sh.a[s], ta, kb * kLmBK, row0, &sh.full[s]);
                    tma_load_2d(sh.b[s], &tmB, kb * kLmBK, n_blk * kLmBN, &sh.full[s]);
                }
            }
            // teardown: let the last copy of every stage land before the CTA exits
            for (int s = 0; s < kLmStages; ++s) {
                const uint32_t n = it / kLmStages + ((uint32_t)s < it % kLmStages ? 1u : 0u);
                if (n > 0) mbar_wait_bounded(&sh.full[s], (n - 1) & 1u, kLmWaitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------------------------------- MMA issuer
            uint32_t it = 0, tcount = 0;
            for (int tile = blockIdx.x; tile < num_tiles && !*abort; tile += gridDim.x, ++tcount) {
                const uint32_t buf = tcount & 1u, use = tcount >> 1;
                if (use > 0 && !lm_wait(&sh.acc_empty[buf], (use - 1) & 1u, abort, limit_ns)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + buf * kLmBN;
                bool ok = true;
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const int s = (int)(it % kLmStages);
                    if (!lm_wait(&sh.full[s], (it / kLmStages) & 1u, abort, limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_desc_sw128(smem_u32(sh.a[s]));
                    const uint64_t bd = umma_desc_sw128(smem_u32(sh.b[s]));
#pragma unroll
                    for (int k = 0; k < kLmBK / 16; ++k)  // 16 elements = 32 bytes = 2 units
                        umma_bf16(d_tmem, ad + 2u * k, bd + 2u * k, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(&sh.empty[s]);  // the stage is free once these MMAs are done
                }
                if (!ok) break;
                umma_commit(&sh.acc_full[buf]);  // the accumulator is complete
            }
            // teardown: every MMA issued has finished before the TMEM is freed
            umma_commit(&sh.done);
            mbar_wait_bounded(&sh.done, 0u, kLmWaitNs);
        }
    } else {  // ------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lanes 32 q .. 32 q + 31 belong to this warp
        const int r_in = q * 32 + lane;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
            const uint32_t buf = tcount & 1u, use = tcount >> 1;
            const bool ok = lm_wait(&sh.acc_full[buf], use & 1u, abort, limit_ns);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int m_blk = tile % m_tiles, n_blk = tile / m_tiles;
            const int seg = m_blk >= mt0 ? 1 : 0;
            const int r = (seg ? m_blk - mt0 : m_blk) * kLmBM + r_in;
            epi.row(seg, r, r < (seg ? M1 : M0), n_blk * kLmBN, V,
                    tmem + ((uint32_t)(q * 32) << 16) + buf * kLmBN);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(reinterpret_cast<unsigned long long *>(&sh.acc_empty[buf]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kLmTmemCols);
    }
    if (threadIdx.x == 0 && sh.abort && status) atomicOr(status, 4u /* SPEC_DEV_TIMEOUT */);
}

} // namespace sv
